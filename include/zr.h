/*
 * zr.h -- C ABI of libzr: partition-aware ZeRO stage-1/2 gradient averaging
 * followed by the sharded AdamW step, on one GPU (sm_103a).
 *
 * The data-parallel group of N ranks is emulated on one device: each rank's
 * gradients, bucket and optimizer shard are separate device buffers, and the
 * collectives become local HBM reductions over those N buffers. Nothing
 * crosses GPUs; the library issues no collective and links no communication
 * library.
 *
 * Sources, cited by page title and section:
 *   [DS] "DeepSpeed ZeRO 通信优化深度解析：用 reduce-scatter 分区感知规约替代 all-reduce"
 *   [MG] "Megatron-LM 分布式训练（四）：数据并行 DP 与分布式优化器（ZeRO）"
 *   [IQ] "07. 大规模训练时通信瓶颈在哪里？AllReduce、AllGather、ReduceScatter 有什么区别？"
 *
 * Notation: N = world, n_i = numel of param i, o_i = sum_{j<i} n_j,
 * T = sum n_i, P = ceil(T/N)*N (tail padding only), S = P/N; rank r owns the
 * flat range [rS, (r+1)S).
 *
 * Conventions for every entry point:
 *  - Returns ZR_OK (0) or a negative ZR_ERR_* status; zr_last_error() gives
 *    a message for the calling thread's last failure. The library never
 *    throws across this boundary, never exits or aborts, and its kernels
 *    never trap.
 *  - Device buffers are owned by the caller. The library allocates the
 *    host-side layout handle (freed by zr_layout_destroy) and, in device
 *    memory, only the tables of a plan (zr_pack_plan_create,
 *    zr_direct_plan_create; freed by the matching destroy), the sums of a
 *    gradient check (zr_gradcheck_create) and the counters of
 *    zr_arith_check; the other kernels take their tables as launch
 *    parameters and use no scratch memory.
 *  - Kernels may read, never write, bytes that share an aligned 16-byte chunk
 *    with an element of an input tensor (they move whole aligned chunks);
 *    such a chunk never crosses a page, so this cannot fault.
 *  - "host array of device pointers": a host array (read during the call
 *    only) whose entries are device addresses.
 *  - A device address may point into pinned (page-locked) host memory, which
 *    the CUDA runtime maps into the device's address space at the same
 *    address: the kernels then read or write it in place over the host link
 *    (for example a direct plan over host-resident gradients, with the bf16
 *    parameters written to a pinned host buffer), at the link's bandwidth.
 *  - Kernels are enqueued on `stream` (NULL = the legacy default stream) and
 *    the call returns without synchronising. Launch errors are reported;
 *    errors of the asynchronous execution surface at the caller's next
 *    synchronisation.
 *  - Device pointers need only element alignment (2 bytes for bf16, 4 for
 *    fp32); otherwise ZR_ERR_ALIGN. Any 16-byte phase is accepted. The fused
 *    steps run fastest when partition r of master, m and v (and of the shard
 *    gradient) starts at the same 16-byte phase, modulo 4 elements, as element
 *    r*S of param_bf16: as views at offset r*S of flat [P] buffers laid out
 *    like the parameters. Their tiles then start every stream on a 16-byte
 *    boundary; results are the same either way.
 *  - Outputs must not overlap inputs except where an argument is in/out.
 */
#ifndef ZR_H
#define ZR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZR_OK 0
#define ZR_ERR_INVALID_ARG (-1)  /* NULL, out-of-range index, bad size or dtype */
#define ZR_ERR_CUDA (-2)         /* a CUDA runtime call or launch failed */
#define ZR_ERR_OOM (-3)          /* host allocation failed */
#define ZR_ERR_ALIGN (-4)        /* a device pointer is not element-aligned */
#define ZR_ERR_TIMEOUT (-5)      /* reserved: a bounded device wait ran out */
#define ZR_ERR_STATE (-6)        /* no usable CUDA device / wrong device state */
#define ZR_ERR_UNSUPPORTED (-7)  /* a size beyond what the library supports */

/* Largest world (emulated data-parallel size) the kernels accept. */
#define ZR_MAX_WORLD 1024

/* Defaults of the zero_optimization keys ([DS] §五 table). */
#define ZR_DEFAULT_REDUCE_BUCKET_SIZE 500000000LL
#define ZR_DEFAULT_REDUCE_SCATTER 1
#define ZR_DEFAULT_CONTIGUOUS_GRADIENTS 1
#define ZR_DEFAULT_OVERLAP_COMM 0

typedef struct CUstream_st *zr_stream; /* the same type as cudaStream_t */
typedef struct zr_layout zr_layout;    /* opaque, host-owned */

/* Gradient element types: bf16, fp32, or fp16 (IEEE binary16, the fp16
 * training the pages' all-reduce path scales for, [DS] §三.2, §六). Every
 * value is widened to fp32 exactly before any arithmetic. */
typedef enum { ZR_BF16 = 0, ZR_FP32 = 1, ZR_FP16 = 2 } zr_dtype;

typedef struct {
    int64_t T, P, S;               /* total, padded total, partition size */
    int64_t n_params, n_buckets, n_slices, n_runs;
    int64_t reduce_bucket_size;
    int32_t world;
} zr_layout_info;

/* One (param, partition) intersection ([DS] §三.2: a param's grad cut by
 * destination partition into (dst_rank, bucket_offset, numel) pieces). */
typedef struct {
    int64_t param, bucket;
    int32_t dst;
    int64_t param_offset;      /* grad_start_offset: offset inside the param's grad */
    int64_t bucket_offset;     /* offset inside the bucket */
    int64_t partition_offset;  /* offset inside rank dst's partition */
    int64_t numel;
} zr_slice;

/* Slices of one bucket aimed at one rank, merged ([DS] §三.2: contiguous
 * fragments for the same target are reduced together); the tail padding is
 * part of the last bucket's runs. */
typedef struct {
    int64_t bucket;
    int32_t dst;
    int64_t bucket_offset, partition_offset, numel;
} zr_run;

/* AdamW hyper-parameters; step is the 1-based step count t. */
typedef struct {
    float lr, beta1, beta2, eps, weight_decay;
    int64_t step;
} zr_adamw;

/* The fp32 scalars one AdamW step uses, each computed on the host in double
 * from the fp32 hyper-parameters and rounded once. */
typedef struct {
    float beta1, one_minus_beta1, beta2, one_minus_beta2;
    float step_size;  /* lr / (1 - beta1^t) */
    float bc2_sqrt;   /* sqrt(1 - beta2^t) */
    float decay;      /* 1 - lr * weight_decay */
    float eps;
} zr_adamw_scalars;

/* ---- status ------------------------------------------------------------ */

const char *zr_status_string(int status);
/* Copies the calling thread's last error message (NUL-terminated, truncated
 * to cap). Returns the full message length. */
int zr_last_error(char *buf, size_t cap);
int zr_version(void);
/* Number of kernels this process has launched through libzr so far (all
 * threads, all devices); lets a caller count the launches of a region.
 * Failure injection for testing a caller's error handling: while the
 * environment variable ZR_FAIL_AT_LAUNCH holds n >= 1, every kernel launch
 * attempted once this count has reached n - 1 fails with ZR_ERR_CUDA (message
 * "injected failure ...") before anything is enqueued; the entry point returns
 * at that launch, so later launches of the same call are not made. The
 * variable is read at every attempt; unset or 0, it has no effect. */
int64_t zr_launch_count(void);

/* Whether the current device reaches host address p at the same address (the
 * condition for passing it where the library takes device pointers): *mapped
 * = 1 if the CUDA runtime reports p's device address as p itself (pinned host
 * memory it has mapped; on systems whose device uses the host's page tables,
 * any host memory), 0 otherwise. Returns ZR_ERR_INVALID_ARG if mapped is
 * NULL, else ZR_OK; a refused lookup is not left behind as a pending error. */
int zr_host_mapped(const void *p, int32_t *mapped);

/* ---- layout (host only) ------------------------------------------------ */

/*
 * Builds the flat partitioned layout of n_params parameters of numel[i] >= 1
 * elements each, for `world` ranks (1..ZR_MAX_WORLD), with buckets of at most
 * reduce_bucket_size >= 1 elements.
 *  - Flat layout: params concatenated in order, padded at the tail to a
 *    multiple of world, split in world equal partitions ([DS] §二; [MG]
 *    §"分布式优化器": each card keeps 1/DP of the optimizer state).
 *  - Buckets: params in ascending order; a bucket is closed before a param
 *    that would overflow it, so an oversized param sits alone; the last
 *    bucket also covers the padding [T, P) ([DS] §四, reduce_bucket_size; §五).
 * n_params = 0 gives an empty layout (T = P = S = 0, no buckets).
 * *out is owned by the caller and freed with zr_layout_destroy.
 */
int zr_layout_create(const int64_t *numel, int64_t n_params, int32_t world,
                     int64_t reduce_bucket_size, zr_layout **out);

/*
 * The same layout when the grads arrive in another order than the flat one:
 * arrival[k] is the param whose grad is produced k-th (a permutation of
 * 0..n_params-1; NULL = the flat order, as zr_layout_create). Backward
 * produces the last layers' grads first, and each grad is copied into the
 * IPG bucket as soon as it is produced ([DS] §四), so the buckets fill in
 * arrival order under the same closing rule; the flat layout and the
 * partitions do not change. Param i then sits at its own position inside its
 * bucket (the elements of the params that arrived before it into the same
 * bucket), the tail padding is reduced with the bucket that holds the last
 * flat param (after that bucket's params), and a run is a maximal stretch of
 * a bucket that is also one stretch of one partition ([DS] §三.2: only
 * contiguous fragments aimed at one rank are merged). Every entry point
 * below accepts such a layout; results are bit-identical to the flat order's.
 * ZR_ERR_INVALID_ARG if arrival is not a permutation.
 */
int zr_layout_create_ordered(const int64_t *numel, int64_t n_params, int32_t world,
                             int64_t reduce_bucket_size, const int64_t *arrival, zr_layout **out);
int zr_layout_destroy(zr_layout *layout);
int zr_layout_query(const zr_layout *layout, zr_layout_info *info);

/* param_to_partition_ids and grad_start_offset of one param ([DS] §三.2).
 * Writes min(cap, count) entries (either array may be NULL) and the count. */
int zr_layout_param_partitions(const zr_layout *layout, int64_t param, int32_t *part_ids,
                               int64_t *grad_start_offset, int32_t cap, int32_t *n_out);
/* All slices (param order, then dst) / runs (bucket order, then bucket
 * offset; in the flat order that is also dst order). Writes min(cap, count)
 * entries (out may be NULL to query the count). A slice's bucket_offset is
 * its position in its bucket. */
int zr_layout_slices(const zr_layout *layout, zr_slice *out, int64_t cap, int64_t *n_out);
int zr_layout_runs(const zr_layout *layout, zr_run *out, int64_t cap, int64_t *n_out);
/* Flat start and element count (padding included) of bucket b. The flat
 * start is -1 when the bucket is not one flat range in flat order (an arrival
 * order other than the flat one). */
int zr_layout_bucket(const zr_layout *layout, int64_t b, int64_t *flat_start, int64_t *numel);
/* Flat offset o_i of param i and the bucket it belongs to. */
int zr_layout_param(const zr_layout *layout, int64_t param, int64_t *flat_offset, int64_t *bucket);
/* Where each param's gradient starts inside its bucket, the offset at which
 * zr_bucket_pack places it ([DS] §四: grads copied into the IPG bucket as they
 * arrive): o_i minus the bucket's flat start under the flat arrival order,
 * else the elements of the params that arrived before it into the same
 * bucket. Writes min(cap, n_params) entries to out (may be NULL to query the
 * count) and n_params to *n_out. A caller that reads packed buckets per param
 * (for instance a zr_direct_plan over the bucket buffers' param slices)
 * points into them with these offsets. */
int zr_layout_bucket_positions(const zr_layout *layout, int64_t *out, int64_t cap, int64_t *n_out);

/* ---- device steps ------------------------------------------------------ */

/*
 * IPG bucket packing ([DS] §四: each param's grad is copied into the
 * contiguous reduce_bucket_size bucket; §五 contiguous_gradients).
 * grads: host array [world * n_params] of device pointers, entry k*n_params+i
 *   = replica k's grad of param i (numel[i] elements of dtype); only the
 *   params of `bucket` are read (others may be NULL).
 * bucket_out: host array [world] of device pointers, each receiving numel_b
 *   elements: param i's element e at offset o_i - bucket_start + e, and zeros
 *   at positions past T (the padding of the last bucket).
 * The bucket is one buffer per emulated rank (each rank owns separate memory)
 * rather than one [world][numel_b] buffer; a caller holding one such buffer
 * passes the addresses of its rows.
 */
int zr_bucket_pack(const zr_layout *layout, int64_t bucket, const void *const *grads,
                   zr_dtype dtype, void *const *bucket_out, zr_stream stream);

/*
 * A pack plan: the segment descriptors of every bucket of `layout` for one set
 * of gradient tensors and bucket buffers (same arguments as zr_bucket_pack),
 * uploaded once to device memory so that each bucket is packed by a single
 * launch. Training loops keep their gradient and bucket tensors across steps,
 * so the plan is built once and reused; rebuild it if any pointer changes.
 * The plan allocates device memory on the current device (about 48 bytes per
 * (replica, param) pair) and copies to it synchronously; it holds the pointers
 * it was given, not the tensors. Same packing semantics as zr_bucket_pack.
 */
typedef struct zr_pack_plan zr_pack_plan;
int zr_pack_plan_create(const zr_layout *layout, const void *const *grads, zr_dtype dtype,
                        void *const *bucket_out, zr_pack_plan **out);
int zr_pack_plan_destroy(zr_pack_plan *plan);
/* Packs bucket b of the plan: one kernel launch on `stream`. */
int zr_bucket_pack_planned(const zr_pack_plan *plan, int64_t bucket, zr_stream stream);

/*
 * zr_bucket_pack without any device allocation, for callers that cannot call
 * cudaMalloc: for example a framework that serves all device memory from its
 * own pool and holds the process to a fixed budget, where an allocation behind
 * its back would break the budget or fail. The pages have no counterpart to
 * this; it is a deployment convenience.
 * Same arguments and results as zr_bucket_pack, in one packing launch: the
 * bucket's segment table (one segment per replica and param, contiguous params
 * merged, plus the padding) is written into a fixed table inside the library's
 * device code, at most 8192 segments (384 KB, held on every GPU that loads the
 * library until exit), by small kernels that carry up to 600 segments each in
 * their launch parameters. Nothing is copied from host memory, so the call
 * does not wait for the stream. A bigger bucket returns ZR_ERR_UNSUPPORTED.
 * The first call on a device looks the table's address up
 * (cudaGetSymbolAddress). All calls share the table: calls on one stream are ordered, but calls whose work
 * overlaps on the GPU (different streams) race on it.
 */
int zr_bucket_pack_noalloc(const zr_layout *layout, int64_t bucket, const void *const *grads, zr_dtype dtype,
                           void *const *bucket_out, zr_stream stream);

/*
 * fp32 main-grad accumulation ([MG] §"四步接力" step 2: main_grad.add_(grad)
 * into the fp32 contiguous buffer): main_grad[e] += float(g[e]), e < n.
 * main_grad: device fp32 [n], in/out. g: device [n] of g_dtype.
 */
int zr_grad_accumulate(float *main_grad, const void *g, zr_dtype g_dtype, int64_t n,
                       zr_stream stream);

/*
 * The first micro-step of an accumulation: main_grad[e] = 0 + float(g[e]),
 * the value zr_grad_accumulate gives on a zeroed buffer (0 + -0 is +0),
 * without reading main_grad or zeroing it first.
 */
int zr_grad_accumulate_first(float *main_grad, const void *g, zr_dtype g_dtype, int64_t n,
                             zr_stream stream);

/*
 * Reduce-scatter with average over one bucket ([DS] §三.2 and §六: predivide
 * by the data-parallel size, then reduce each slice to its owner; [IQ]
 * §"三种原语": GPU i gets segment i of the sum; [DS] §三.3
 * copy_grads_in_partition).
 * For every bucket position e (flat f = bucket_start + e, owner r = f / S):
 *   shard_grad[r][f - rS] = sum over k = 0..world-1, in that order, of
 *                           fp32(bucket_in[k][e]) * scale, summed in fp32.
 * bucket_in: host array [world] of device pointers, numel_b elements each.
 * scale: the predivide factor, normally 1/world (dp_world_size/sp_size per
 *   [DS] §六); any finite value.
 * shard_grad: host array [world] of device pointers, S fp32 each; only the
 *   entries of ranks the bucket intersects are read, only positions inside
 *   the bucket are written.
 * bucket_in is a host array of one buffer per rank rather than one
 * [world][numel_b] buffer (pass its rows' addresses to use one).
 */
int zr_reduce_scatter_avg(const zr_layout *layout, int64_t bucket, const void *const *bucket_in,
                          zr_dtype dtype, float scale, float *const *shard_grad, zr_stream stream);

/*
 * zr_reduce_scatter_avg for the buckets [bucket_first, bucket_first +
 * bucket_count) of one contiguous gradient buffer per rank ([DS] §五
 * contiguous_gradients: the gradients are copied into one contiguous buffer;
 * [MG] §"梯度缓冲区+分桶+overlap": the flat gradient buffer is cut into buckets
 * that are reduce-scattered in turn). grad_buf[k]: host array [world] of device
 * pointers; rank k's buffer holds every bucket back to back in bucket order,
 * bucket b at element offset numel_0 + ... + numel_{b-1} (in the flat arrival
 * order that is the flat layout itself, padding last: the [P] gradient buffer);
 * only the range's buckets are read. Consecutive buckets share launches up to
 * 2^26 elements, and the results equal one zr_reduce_scatter_avg call per
 * bucket (bucket_in[k] = grad_buf[k] + that offset), bit for bit.
 * Differs from the per-bucket call only in where the buckets sit: one buffer
 * per rank for the whole range instead of one bucket buffer per call.
 * Stream order as for zr_step_direct_range: the first launch waits for all
 * earlier work; later launches of the call (other runs, other outputs) may
 * start while the one before drains, and complete only after it.
 */
int zr_reduce_scatter_avg_range(const zr_layout *layout, int64_t bucket_first, int64_t bucket_count,
                                const void *const *grad_buf, zr_dtype dtype, float scale,
                                float *const *shard_grad, zr_stream stream);

/*
 * AdamW over whole partitions ([MG] §"通信模式": each card updates its own
 * 1/DP slice with the fp32 master; §"朴素 DP 的致命浪费": master, m, v are
 * the 12 sharded bytes). Per element, each operation rounded to fp32:
 *   m' = b1 m + (1-b1) g;  v' = b2 v + (1-b2) g^2;
 *   p' = p (1 - lr wd) - (lr/(1-b1^t)) * m' / (sqrt(v')/sqrt(1-b2^t) + eps).
 * master, m, v (in/out) and grad: host arrays [world] of device pointers, S
 * fp32 each. rank in [0, world) updates that rank's shard only (other
 * entries may be NULL); rank = -1 updates every rank.
 */
int zr_adam_shard_step(const zr_layout *layout, int32_t rank, float *const *master,
                       float *const *m, float *const *v, const float *const *grad,
                       const zr_adamw *hp, zr_stream stream);

/*
 * All-gather payload ([MG] §"通信模式": the updated slices are concatenated
 * back into the full weights for the next forward; [IQ] §"三种原语"):
 *   param_bf16[f] = bf16_round_nearest_even(master[f / S][f % S]) for f < T,
 *   param_bf16[f] = 0 for T <= f < P.
 * master: host array [world] of device pointers, S fp32 each.
 * param_bf16: device [P] bf16.
 */
int zr_gather_cast_bf16(const zr_layout *layout, const float *const *master, void *param_bf16,
                        zr_stream stream);

/*
 * The three steps above in one pass over one bucket: the averaged gradient
 * of each position is kept in registers, AdamW updates the owner's master,
 * m and v, and the updated master is cast to bf16 into the full parameter
 * buffer ([MG] §"通信模式": reduce-scatter, then the local fp32 update,
 * then the all-gather's payload). Results are bit-identical to
 * zr_reduce_scatter_avg + zr_adam_shard_step + zr_gather_cast_bf16 restricted
 * to the bucket's positions.
 * param_bf16: device [P] bf16 or NULL (not written).
 * shard_grad_out: host array [world] of device pointers (S fp32 each) or NULL;
 *   if given, it also receives the averaged gradient.
 */
int zr_rs_adam_fused(const zr_layout *layout, int64_t bucket, const void *const *bucket_in,
                     zr_dtype dtype, float scale, float *const *master, float *const *m,
                     float *const *v, const zr_adamw *hp, void *param_bf16,
                     float *const *shard_grad_out, zr_stream stream);

/*
 * zr_rs_adam_fused for the buckets [bucket_first, bucket_first + bucket_count)
 * of one contiguous gradient buffer per rank, laid out as for
 * zr_reduce_scatter_avg_range (grad_buf[k]: rank k's buffer, every bucket back
 * to back in bucket order; only the range's buckets are read). Consecutive
 * buckets share launches up to 2^26 elements, and the results equal one
 * zr_rs_adam_fused call per bucket (bucket_in[k] = grad_buf[k] + the bucket's
 * offset), bit for bit. master, m, v, param_bf16 and shard_grad_out as for
 * zr_rs_adam_fused. Stream order as for zr_reduce_scatter_avg_range.
 */
int zr_rs_adam_fused_range(const zr_layout *layout, int64_t bucket_first, int64_t bucket_count,
                           const void *const *grad_buf, zr_dtype dtype, float scale, float *const *master,
                           float *const *m, float *const *v, const zr_adamw *hp, void *param_bf16,
                           float *const *shard_grad_out, zr_stream stream);

/*
 * zr_rs_adam_fused with the last micro-step's accumulation folded in ([MG]
 * §"四步接力": every micro-step's 16-bit grad is added into the fp32 main_grad
 * before the bucket is reduced; §"通信模式"): for bucket position e,
 *   g_k[e] = fp32(main_in[k][e] + last_in[k][e]),
 * then the averaging, AdamW and cast of zr_rs_adam_fused over the g_k. The
 * results equal zr_grad_accumulate of last_in[k] into main_in[k] followed by
 * zr_rs_adam_fused on main_in, bit for bit, but main_in is only read: the
 * accumulated main_grad is never stored, which saves writing it and reading
 * it back (8 of the 14 bytes per replica and element of the unfused pair).
 * main_in: host array [world] of device pointers, numel_b fp32 each (the
 *   contiguous main_grad buffer's bucket, holding the earlier micro-steps).
 * last_in: host array [world] of device pointers, numel_b elements of
 *   last_dtype (ZR_BF16 or ZR_FP16) each, in the same bucket order.
 * world <= 32 (ZR_ERR_UNSUPPORTED above). Other arguments as for
 * zr_rs_adam_fused.
 */
int zr_rs_adam_fused_acc(const zr_layout *layout, int64_t bucket, const float *const *main_in,
                         const void *const *last_in, zr_dtype last_dtype, float scale, float *const *master,
                         float *const *m, float *const *v, const zr_adamw *hp, void *param_bf16,
                         float *const *shard_grad_out, zr_stream stream);

/*
 * Steps 1 to 4 in one pass, without a bucket buffer. A direct plan records,
 * once, where every replica's gradient of every param of every bucket lives
 * (grads as for zr_bucket_pack; the tensors must stay allocated, at the same
 * addresses, while the plan is used) and how the bucket's elements map to
 * params (in flat order when the bucket holds a contiguous range of params,
 * as under flat or backward arrival: the step needs no bucket buffer, so the
 * order inside a bucket is free, and flat order makes its runs those of the
 * partitions; in bucket order otherwise), in device memory the plan owns (8 bytes per replica and param, 8
 * per param, 36 per 256 bucket positions) plus a host copy of the param
 * offsets. zr_step_direct then does for bucket b what zr_bucket_pack followed
 * by zr_rs_adam_fused does, with identical results: each replica's slice of
 * each param is read where it lies, by its grad_start_offset, instead of
 * being packed first ([DS] §三.2 slicing by param_to_partition_ids /
 * grad_start_offset; [DS] §四). One kernel launch per bucket and per 256
 * runs of it (plus one per further 1,024 tiles that cross a param boundary,
 * when a launch has more).
 * The plan also holds, per bucket, 32 bytes of counters: the warps of a
 * launch that starts at that bucket take their tiles from them as they go
 * (SMs that run faster take more), and the launch leaves them at zero. Calls whose
 * buckets are disjoint may therefore run on different streams at once; calls
 * that share a bucket must be ordered (they write the same elements anyway).
 * The gradients may lie in pinned (page-locked, mapped) host memory instead
 * of device memory, and param_bf16 likewise: the kernels then read and write
 * them over the host link, with no copy. A plan whose rank-0 first gradient
 * is such host memory (as the runtime reports it at creation) runs its steps
 * on plain loads, which draw the host link's rate; device plans run on the
 * copy pipeline, except the step at world <= 2. Which kernel runs changes no
 * result.
 * world <= 32 (ZR_ERR_UNSUPPORTED above).
 * master, m, v, shard_grad_out, param_bf16: as for zr_rs_adam_fused.
 */
typedef struct zr_direct_plan zr_direct_plan;
int zr_direct_plan_create(const zr_layout *layout, const void *const *grads, zr_dtype dtype,
                          zr_direct_plan **out);
int zr_direct_plan_destroy(zr_direct_plan *plan);
int zr_step_direct(const zr_direct_plan *plan, int64_t bucket, float scale, float *const *master,
                   float *const *m, float *const *v, const zr_adamw *hp, void *param_bf16,
                   float *const *shard_grad_out, zr_stream stream);

/*
 * zr_step_direct for buckets [bucket_first, bucket_first + bucket_count), in
 * few launches: consecutive buckets share one while their runs, their tables
 * and their boundary tiles fit the launch parameters (256 runs, 16 buckets and
 * 1,024 listed tiles) and the launch stays within 2^26 elements; a longer run
 * gets a launch of its own. The buckets' elements are disjoint, so
 * the results equal bucket_count calls of zr_step_direct bit for bit; longer
 * launches spend less of their time filling and draining the pipelines. For
 * a step that runs once every bucket's gradients are ready (after backward,
 * or at a gradient-accumulation boundary); a step that reduces buckets as
 * backward fills them calls zr_step_direct per bucket.
 * Stream order: the call's first launch starts after all earlier work on
 * the stream, as any launch does. Each later launch of the same call (other
 * buckets, other tile counters) is a programmatic dependent of the one
 * before: its blocks may start while that launch drains, and it completes
 * only after that launch has. So work queued after the call, and an event
 * recorded after it, still see the whole call complete; in between, the
 * call's launches overlap.
 */
int zr_step_direct_range(const zr_direct_plan *plan, int64_t bucket_first, int64_t bucket_count, float scale,
                         float *const *master, float *const *m, float *const *v, const zr_adamw *hp,
                         void *param_bf16, float *const *shard_grad_out, zr_stream stream);

/*
 * All-reduce with average over one bucket, the path used when
 * reduce_scatter is off ([DS] §三.2 gradient_reduction_w_predivide; [MG]
 * §"四步接力" step 4; [IQ] §"三种原语"): out[k][e] = the same averaged value
 * as zr_reduce_scatter_avg, then multiplied by `postscale` (fp32, rounded),
 * for every replica k. That path keeps fp16 training's pre- and post-scaling
 * ([DS] §三.2 gradient_predivide_factor and postscale_gradients; §六 "divide
 * first"): with predivide factor f, scale = 1/f and postscale = f/N; f = N
 * means postscale = 1, which leaves the average unchanged bit for bit.
 * out: host array [world] of device pointers, numel_b fp32 each.
 * ZR_ERR_INVALID_ARG if postscale is not finite.
 * bucket_in and out are host arrays of one buffer per rank rather than one
 * [world][numel_b] buffer each, and postscale is an argument of its own
 * (1.0f for the plain average).
 */
int zr_allreduce_avg(const zr_layout *layout, int64_t bucket, const void *const *bucket_in,
                     zr_dtype dtype, float scale, float postscale, float *const *out, zr_stream stream);

/*
 * zr_allreduce_avg over the buckets [bucket_first, bucket_first + bucket_count)
 * of one contiguous gradient buffer per rank, laid out as for
 * zr_reduce_scatter_avg_range; out[k] (host array [world] of device pointers,
 * fp32) receives the same bucket-order layout, and only the range's positions
 * are written. Consecutive buckets share launches up to 2^26 elements; the
 * results equal one zr_allreduce_avg call per bucket, bit for bit. The
 * averaging launches overlap as in zr_reduce_scatter_avg_range; the copy to
 * the other replicas starts after the last of them has completed.
 */
int zr_allreduce_avg_range(const zr_layout *layout, int64_t bucket_first, int64_t bucket_count,
                           const void *const *grad_buf, zr_dtype dtype, float scale, float postscale,
                           float *const *out, zr_stream stream);

/* ---- global gradient check before the step -------------------------------- */

/*
 * Between the DP sync of every bucket and optimizer.step() ([MG]
 * §"跨 model-parallel 的梯度收尾": DP sync first, then the remaining gradient
 * fix-ups, then the step; [DS] §六: fp16 training guards its gradient
 * arithmetic): the global L2 norm of the averaged gradient over every rank's
 * partition, an overflow check, and clipping by that norm. The pages give no
 * formula; the usual one is taken:
 *   sumsq     = the sum of g^2 over every rank's shard gradient;
 *   norm      = sqrt(sumsq);
 *   nonfinite = the number of elements whose fp32 square g*g is not finite;
 *   skip      = nonfinite > 0: the step changes nothing (an overflowed step
 *               is dropped, as fp16 loss scaling does; the loss scale is
 *               the caller's, and 1/loss_scale may be folded into `scale`);
 *   coef      = fp32(min(1, max_norm / (norm + 1e-6))) when max_norm > 0
 *               and not skip, else 1.
 * The check needs the whole gradient before any element's update, so the
 * step takes two passes: the averaging of every bucket into the shard
 * gradients (zr_rs_direct_norm or zr_reduce_scatter_avg_norm, which also add
 * to the check's sums), then zr_grad_check_finalize and zr_adam_clip_step.
 * The outcome stays in device memory (no host round trip) until
 * zr_gradcheck_read.
 *
 * Accuracy: a thread adds the fp32 squares of its 8 elements of a tile in
 * fp32 and the result to a double (a square outside [2^-100, 2^100] goes to
 * the double exactly), so sumsq is within about 1e-6 relative of the exact
 * sum. The blocks' sums are added in a fixed order, so the outcome repeats
 * exactly for the same inputs and launch sequence on the same device when
 * the calls that add to one check are ordered (one stream, or events);
 * concurrent calls still add correctly, in some order.
 */
typedef struct {
    double sumsq;        /* the sum of squares */
    double norm;         /* sqrt(sumsq) */
    uint64_t nonfinite;  /* averaged gradients whose fp32 square is not finite */
    float coef;          /* the clip coefficient the step applies */
    int32_t skip;        /* 1: the step leaves every state unchanged */
} zr_grad_stats;

typedef struct zr_gradcheck zr_gradcheck;

/* Allocates on the current device the check's sums (65,536 per-block slots
 * and the finalize's scratch, about 1 MB, zeroed) and its outcome (coef = 1,
 * skip = 0 until the first finalize). */
int zr_gradcheck_create(zr_gradcheck **out);
int zr_gradcheck_destroy(zr_gradcheck *chk);

/* Clears the sums (after a step abandoned before its finalize). */
int zr_gradcheck_reset(zr_gradcheck *chk, zr_stream stream);

/*
 * zr_reduce_scatter_avg over one packed bucket, also adding the averages'
 * squares and non-finite count to chk.
 */
int zr_reduce_scatter_avg_norm(const zr_layout *layout, int64_t bucket, const void *const *bucket_in,
                               zr_dtype dtype, float scale, float *const *shard_grad, zr_gradcheck *chk,
                               zr_stream stream);

/*
 * The direct plan's pass without the optimizer: every replica's gradients of
 * bucket b, read where they lie, averaged into shard_grad exactly as
 * zr_bucket_pack followed by zr_reduce_scatter_avg would, adding to chk.
 * shard_grad: host array [world] of device pointers, S fp32 each (the
 * entries of the ranks the bucket intersects). world <= 32.
 */
int zr_rs_direct_norm(const zr_direct_plan *plan, int64_t bucket, float scale, float *const *shard_grad,
                      zr_gradcheck *chk, zr_stream stream);

/* zr_rs_direct_norm for buckets [bucket_first, bucket_first + bucket_count),
 * grouped into launches as zr_step_direct_range groups them, with the same
 * stream order (later launches of the call overlap the one before). Each
 * launch adds its sums to chk only after the launch before it has completed,
 * so the sums are added in the same order on every call. */
int zr_rs_direct_norm_range(const zr_direct_plan *plan, int64_t bucket_first, int64_t bucket_count, float scale,
                            float *const *shard_grad, zr_gradcheck *chk, zr_stream stream);

/*
 * Once every bucket has been added: sums chk's accumulators in a fixed
 * order, writes the outcome for max_norm (<= 0: no clipping; NaN is
 * ZR_ERR_INVALID_ARG) and clears the accumulators for the next step.
 */
int zr_grad_check_finalize(zr_gradcheck *chk, float max_norm, zr_stream stream);

/*
 * The step the outcome steers, over every rank's shard: nothing if skip;
 * otherwise for every element, gc = grad * coef (fp32, exact when coef = 1),
 * the AdamW update of zr_adam_shard_step with gc, and the bf16 cast of
 * zr_gather_cast_bf16 into param_bf16 ([MG] §"通信模式"). With max_norm <= 0
 * and finite gradients the results equal those of zr_rs_adam_fused bit for
 * bit. master, m, v (in/out) and grad: host arrays [world] of device
 * pointers, S fp32 each. param_bf16: device [P] bf16 or NULL.
 */
int zr_adam_clip_step(const zr_layout *layout, float *const *master, float *const *m, float *const *v,
                      const float *const *grad, const zr_adamw *hp, const zr_gradcheck *chk,
                      void *param_bf16, zr_stream stream);

/* Waits for `stream`, then copies the last finalized outcome to *out. */
int zr_gradcheck_read(const zr_gradcheck *chk, zr_stream stream, zr_grad_stats *out);

/* ---- arithmetic self-check (device) -------------------------------------- */

/*
 * Compares, on the current device, the arithmetic the AdamW kernels use
 * with CUDA's IEEE-754 operations (sqrt.rn, rcp.rn, div.rn). The kernels
 * take the square root and the two divisions of the AdamW update ([DS]
 * §四; torch.optim.AdamW's order of operations) through the hardware's
 * approximate reciprocal (square root) and exact fma residuals (Markstein's
 * method); this checks that they round as the IEEE operations do. The pages
 * have no counterpart: it is a check of this library's arithmetic.
 *   which 0: sqrt of every float bit pattern in [begin, begin + count) that
 *            lies where the kernels take the fma route (+0, [2^-100, FLT_MAX]);
 *         1: reciprocal of every bit pattern in [begin, begin + count) whose
 *            magnitude lies in [2^-60, 2^60] (the divisors that route sees);
 *         2: count random quotients a / b drawn by splitmix64 from index
 *            begin + i, a = +0 or |a| in [2^-60, 2^61), b in [2^-60, 2^60],
 *            each with a second, near-exact pair a = RN(b q);
 *         3: count random AdamW elements (p, m, v, g over several decades,
 *            including ones outside that route) under `hp`, compared with the
 *            element computed by the IEEE operations (p, m and v bit for bit).
 * For which 0 and 1, begin + count <= 2^32. hp is read for which 3 only.
 * Writes the mismatch count to *mismatches and up to min(n_bad, 8) of the
 * offending indices to bad (may be NULL). Allocates a few bytes of device
 * memory and blocks until the check is done (device-wide synchronize).
 */
int zr_arith_check(int32_t which, uint64_t begin, uint64_t count, const zr_adamw *hp,
                   uint64_t *mismatches, uint64_t *bad, int32_t n_bad);

/* ---- bounds-checked build ------------------------------------------------ */

/*
 * The library also builds as libzr_checked.so (compiled with ZR_CHECKED),
 * with the same entry points. There, every range a kernel takes from its
 * launch's plan for its vector accesses is checked before the access (a tile
 * inside its run, a replica's tile inside its param's gradient, a packing
 * super-tile inside its segment, a listed element's param inside the
 * bucket); a failed check skips that access or takes the element-by-element
 * path instead, and is counted on the device. The pages have no counterpart:
 * it is a check of this library's planning, for tests (no GPU has to fault).
 * zr_debug_checks waits for the device, then gives the number of failed
 * checks since the last reset, the first one's check code and element, and
 * with reset != 0 clears them. Any pointer may be NULL. In the ordinary
 * build it returns ZR_ERR_UNSUPPORTED.
 */
int zr_debug_checks(int32_t reset, uint64_t *count, int32_t *first_code, int64_t *first_where);

/* ---- accounting (host only) -------------------------------------------- */

/* The AdamW scalars the kernels use for `hp` (see zr_adamw_scalars). */
int zr_adamw_prepare(const zr_adamw *hp, zr_adamw_scalars *out);

/*
 * Bytes one rank sends per step over the padded flat buffer, ring
 * collectives ([MG] §"NCCL 底层算法": 2(N-1)/N of the message per card for a
 * ring all-reduce; [DS] §一: 1.5x -> 1.0x of data parallelism):
 *   scheme 0 DP all-reduce 2(N-1)S e; 1 first ZeRO-1 (all-reduce + all-gather)
 *   3(N-1)S e; 2 partition-aware (reduce-scatter + all-gather) 2(N-1)S e;
 *   3 reduce-scatter only (N-1)S e.
 */
int zr_comm_bytes(const zr_layout *layout, int32_t scheme, int32_t elem_bytes,
                  double *per_rank_bytes);

/*
 * Per-rank bytes of weights, grads and optimizer state ([MG] §"朴素 DP 的致命
 * 浪费": 2+2+4+4+4 = 16 per param; §"ZeRO 各档" table): stage 0 16T;
 * stage 1 4T + 12S; stage 15 (ZeRO-1.5 / stage 2) 2T + 14S; stage 3 16S.
 */
int zr_layout_bytes(const zr_layout *layout, int32_t stage, double *bytes_per_rank);

#ifdef __cplusplus
}
#endif

#endif /* ZR_H */

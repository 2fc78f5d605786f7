/*
 * zr_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of what partition-aware ZeRO
 * stage-1/2 gradient averaging followed by the sharded AdamW step computes.
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline may load this file. The product library never links, includes or
 * calls it, and the two share no source, header, table or helper.
 *
 * Sources, cited by page title and section:
 *   [DS] "DeepSpeed ZeRO 通信优化深度解析：用 reduce-scatter 分区感知规约替代 all-reduce"
 *   [MG] "Megatron-LM 分布式训练（四）：数据并行 DP 与分布式优化器（ZeRO）"
 *   [IQ] "07. 大规模训练时通信瓶颈在哪里？AllReduce、AllGather、ReduceScatter 有什么区别？"
 *
 * Notation: N = world, n_i = numel of param i, o_i = sum_{j<i} n_j,
 * T = sum n_i, P = ceil(T/N)*N, S = P/N; partition r is flat [rS, (r+1)S).
 *
 * Build: cc -std=c99 -O2 -ffp-contract=off -fPIC -shared. No FMA contraction:
 * every floating-point operation below is rounded to fp32 on its own, in the
 * order written.
 *
 * Parity status: every function is pinned by the CPU tests (brute force on
 * tiny layouts, closed forms, a library cross-check or the pages' own tables).
 * No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ZRO_OK 0
#define ZRO_EINVAL (-1)

#define ZRO_BF16 0
#define ZRO_FP32 1
#define ZRO_FP16 2

/* ------------------------------------------------------------------------- */
/* bf16 <-> fp32 by bit pattern                                               */
/* ------------------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32, so widening is exact. */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round-to-nearest-even narrowing of binary32 to bf16, the cast that makes
 * the bf16 weights of [MG] §"朴素 DP 的致命浪费" from the fp32 master.
 * Adds 0x7FFF plus the lowest kept bit, then drops the low 16 bits (ties go
 * to the even neighbour; overflow carries into the exponent, giving inf).
 * NaN becomes the quiet NaN 0x7FC0. */
static uint16_t f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)0x7FC0;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* IEEE 754 binary16 widened to binary32, exactly: sign, 5-bit exponent of
 * bias 15, 10-bit fraction; exponent 0 holds zero and the subnormals
 * (fraction x 2^-24), exponent 31 the infinities and NaNs (payload kept).
 * The fp16 gradients of the pages' fp16 training ([DS] §三.2, §六). */
static float f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) << 31, e = (h >> 10) & 0x1fu, fr = h & 0x3ffu, u;
    float f;
    if (e == 0) {
        f = ldexpf((float)fr, -24);  /* exact: fr < 2^10 */
        memcpy(&u, &f, sizeof u);
        u |= sign;
    } else if (e == 31) {
        u = sign | 0x7F800000u | (fr << 13);
    } else {
        u = sign | ((e - 15u + 127u) << 23) | (fr << 13);
    }
    memcpy(&f, &u, sizeof f);
    return f;
}

void zro_f16_to_f32(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f16_to_f32(in[i]);
}

static float load_elem(const void *base, int32_t dtype, int64_t i)
{
    if (dtype == ZRO_BF16) return bf16_to_f32(((const uint16_t *)base)[i]);
    if (dtype == ZRO_FP16) return f16_to_f32(((const uint16_t *)base)[i]);
    return ((const float *)base)[i];
}

void zro_bf16_to_f32(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_f32(in[i]);
}

void zro_f32_to_bf16(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(in[i]);
}

/* ------------------------------------------------------------------------- */
/* Flat partitioned layout, buckets, slices and merged runs                    */
/* ------------------------------------------------------------------------- */

static int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
static int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

/*
 * Builds the whole layout. Every output pointer may be NULL (then it is only
 * counted). dims = {T, P, S, n_buckets, n_slices, n_runs}.
 *
 * Flat layout: the parameters are concatenated in order, the total is padded
 *   at the tail to a multiple of N and split into N equal partitions; rank r
 *   owns the r-th ([DS] §二: optimizer state and 16-bit grads are cut into
 *   data-parallel-degree equal parts, each rank holding one; [MG]
 *   §"分布式优化器": every card is responsible for 1/DP).
 * Buckets: the parameters, in ascending order, fill a bucket of at most
 *   bucket_size elements; a bucket is closed before a parameter that would
 *   overflow it, so an oversized parameter sits alone; the last bucket also
 *   covers the tail padding ([DS] §四, the IPG bucket of reduce_bucket_size
 *   elements, flushed when full or at the end of backward; §五 table).
 * Slices: one per (param, partition) intersection: the destination rank, the
 *   offset inside the param's grad where the slice starts (grad_start_offset),
 *   its offset in the bucket and in the partition, and its length ([DS] §三.2,
 *   param_to_partition_ids, grad_start_offset, (dst_rank, bucket_offset, numel)).
 * Runs: adjacent slices of one bucket with the same destination merged into
 *   one, the padding appended to the run it continues ([DS] §三.2: contiguous
 *   fragments of a bucket aimed at the same rank are merged before a single
 *   reduction).
 *
 * offset[n], bucket_of[n], bucket_range[nb][2] = {flat start, flat end},
 * slice[ns][7] = {param, bucket, dst, param_offset, bucket_offset, partition_offset, numel},
 * run[nr][5]   = {bucket, dst, bucket_offset, partition_offset, numel}.
 */
int zro_layout(const int64_t *numel, int64_t n, int32_t world, int64_t bucket_size,
               int64_t *dims, int64_t *offset, int64_t *bucket_of,
               int64_t *bucket_range, int64_t *slice, int64_t *run)
{
    if (n < 0 || world < 1 || bucket_size < 1) return ZRO_EINVAL;
    if (n > 0 && numel == NULL) return ZRO_EINVAL;
    for (int64_t i = 0; i < n; ++i)
        if (numel[i] < 1) return ZRO_EINVAL;

    /* offsets and sizes */
    int64_t T = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (offset) offset[i] = T;
        T += numel[i];
    }
    int64_t P = ((T + world - 1) / world) * world;
    int64_t S = P / world;

    int64_t nb = 0, ns = 0, nr = 0;
    int64_t run_bucket = -1, run_dst = -1, run_end = -1; /* the last run opened */
    int64_t bstart = 0, bcount = 0, o = 0;

    for (int64_t i = 0; i < n; ++i) {
        /* bucket walk */
        if (i == 0) {
            nb = 1;
        } else if (bcount > 0 && bcount + numel[i] > bucket_size) {
            if (bucket_range) { bucket_range[2 * (nb - 1)] = bstart; bucket_range[2 * (nb - 1) + 1] = o; }
            bstart = o;
            bcount = 0;
            ++nb;
        }
        int64_t b = nb - 1;
        if (bucket_of) bucket_of[i] = b;
        bcount += numel[i];

        /* the partitions this param's flat range [o, o + n_i) intersects */
        int64_t r_first = o / S, r_last = (o + numel[i] - 1) / S;
        for (int64_t r = r_first; r <= r_last; ++r) {
            int64_t lo = max64(o, r * S);
            int64_t hi = min64(o + numel[i], (r + 1) * S);
            if (slice) {
                int64_t *s = slice + 7 * ns;
                s[0] = i; s[1] = b; s[2] = r; s[3] = lo - o;
                s[4] = lo - bstart; s[5] = lo - r * S; s[6] = hi - lo;
            }
            ++ns;
            if (run_bucket == b && run_dst == r && run_end == lo - bstart) {
                if (run) run[5 * (nr - 1) + 4] += hi - lo;
            } else {
                if (run) {
                    int64_t *q = run + 5 * nr;
                    q[0] = b; q[1] = r; q[2] = lo - bstart; q[3] = lo - r * S; q[4] = hi - lo;
                }
                ++nr;
            }
            run_bucket = b; run_dst = r; run_end = hi - bstart;
        }
        o += numel[i];
    }

    if (n > 0) {
        /* the last bucket ends at P: the padding [T, P) is reduced with it */
        if (bucket_range) { bucket_range[2 * (nb - 1)] = bstart; bucket_range[2 * (nb - 1) + 1] = P; }
        int64_t b = nb - 1;
        for (int64_t f = T; f < P;) {
            int64_t r = f / S;
            int64_t hi = min64(P, (r + 1) * S);
            if (run_bucket == b && run_dst == r && run_end == f - bstart) {
                if (run) run[5 * (nr - 1) + 4] += hi - f;
            } else {
                if (run) {
                    int64_t *q = run + 5 * nr;
                    q[0] = b; q[1] = r; q[2] = f - bstart; q[3] = f - r * S; q[4] = hi - f;
                }
                ++nr;
            }
            run_bucket = b; run_dst = r; run_end = hi - bstart;
            f = hi;
        }
    }

    if (dims) {
        dims[0] = T; dims[1] = P; dims[2] = S; dims[3] = nb; dims[4] = ns; dims[5] = nr;
    }
    return ZRO_OK;
}

/*
 * The same layout when the grads arrive in another order than the flat one:
 * order[k] is the param whose grad is produced k-th (a permutation of 0..n-1;
 * backward produces the last layers' grads first, and each grad is copied
 * into the IPG bucket as soon as it is produced, [DS] §四). The flat layout
 * and the partitions do not change; only the bucket walk follows arrival:
 *   - buckets fill in arrival order under the same closing rule;
 *   - param i sits at bucket_pos[i] in its bucket: the elements of the params
 *     that arrived before it into the same bucket;
 *   - the tail padding is reduced with the bucket holding the last flat param
 *     (n-1), after that bucket's params;
 *   - a slice's bucket_offset is bucket_pos[i] + (its start - o_i);
 *   - runs: walking a bucket in bucket order, a slice (or padding piece) is
 *     merged into the previous piece when they continue each other both in
 *     the bucket and in the same partition ([DS] §三.2: only contiguous
 *     fragments aimed at one rank are merged).
 * With order[k] = k this is zro_layout.
 * bucket_info[nb][3] = {numel_b, pad_pos (-1: no padding), flat_start (-1
 * unless the bucket is the flat range [flat_start, flat_start + numel_b) in
 * order)}; the other outputs as for zro_layout.
 */
int zro_layout_ordered(const int64_t *numel, int64_t n, int32_t world, int64_t bucket_size,
                       const int64_t *order, int64_t *dims, int64_t *offset, int64_t *bucket_of,
                       int64_t *bucket_pos, int64_t *bucket_info, int64_t *slice, int64_t *run)
{
    if (n < 0 || world < 1 || bucket_size < 1) return ZRO_EINVAL;
    if (n > 0 && (numel == NULL || order == NULL)) return ZRO_EINVAL;
    int64_t *o = (int64_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
    int64_t *bof = (int64_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
    int64_t *pos = (int64_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
    int64_t *seen = (int64_t *)calloc((size_t)(n > 0 ? n : 1), sizeof(int64_t));
    if (!o || !bof || !pos || !seen) { free(o); free(bof); free(pos); free(seen); return -3; }
    int rc = ZRO_OK;
    for (int64_t k = 0; k < n && rc == ZRO_OK; ++k) {
        if (numel[k] < 1 || order[k] < 0 || order[k] >= n || seen[order[k]]) rc = ZRO_EINVAL;
        else seen[order[k]] = 1;
    }
    if (rc != ZRO_OK) { free(o); free(bof); free(pos); free(seen); return rc; }

    int64_t T = 0;
    for (int64_t i = 0; i < n; ++i) { o[i] = T; T += numel[i]; }
    int64_t P = ((T + world - 1) / world) * world;
    int64_t S = P / world;

    /* bucket walk in arrival order */
    int64_t nb = 0, fill = 0;
    for (int64_t k = 0; k < n; ++k) {
        int64_t i = order[k];
        if (k == 0) nb = 1;
        else if (fill > 0 && fill + numel[i] > bucket_size) { ++nb; fill = 0; }
        bof[i] = nb - 1;
        pos[i] = fill;
        fill += numel[i];
    }
    /* each bucket's size, padding position and (when in flat order) flat start */
    int64_t pad_b = n > 0 ? bof[n - 1] : -1;
    for (int64_t b = 0; b < nb; ++b) {
        int64_t size = 0, first = -1, prev = -1, inorder = 1;
        for (int64_t k = 0; k < n; ++k) {
            int64_t i = order[k];
            if (bof[i] != b) continue;
            size += numel[i];
            if (first < 0) first = i;
            else if (i != prev + 1) inorder = 0;
            prev = i;
        }
        int64_t pad_pos = -1;
        if (b == pad_b) {
            pad_pos = size;
            if (prev != n - 1) inorder = 0;
            size += P - T;
        }
        if (bucket_info) {
            bucket_info[3 * b] = size;
            bucket_info[3 * b + 1] = pad_pos;
            bucket_info[3 * b + 2] = inorder ? o[first] : -1;
        }
    }

    /* slices, in param order then partition order */
    int64_t ns = 0;
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t r = o[i] / S; r <= (o[i] + numel[i] - 1) / S; ++r) {
            int64_t lo = max64(o[i], r * S), hi = min64(o[i] + numel[i], (r + 1) * S);
            if (slice) {
                int64_t *sl = slice + 7 * ns;
                sl[0] = i; sl[1] = bof[i]; sl[2] = r; sl[3] = lo - o[i];
                sl[4] = pos[i] + lo - o[i]; sl[5] = lo - r * S; sl[6] = hi - lo;
            }
            ++ns;
        }
    }

    /* runs: each bucket in bucket order (its params in arrival order, then the padding) */
    int64_t nr = 0;
    for (int64_t b = 0; b < nb; ++b) {
        int64_t have = 0, pr = -1, px = 0, pp = 0, pn = 0; /* the open piece */
        for (int64_t k = 0; k <= n; ++k) {
            /* k < n: the k-th arriving param if it is in b; k == n: the padding if b holds it */
            int64_t f0, f1, x0;
            if (k < n) {
                int64_t i = order[k];
                if (bof[i] != b) continue;
                f0 = o[i]; f1 = o[i] + numel[i]; x0 = pos[i];
            } else {
                if (b != pad_b || P == T) break;
                int64_t size_wo_pad = 0;
                for (int64_t q = 0; q < n; ++q) if (bof[q] == b) size_wo_pad += numel[q];
                f0 = T; f1 = P; x0 = size_wo_pad;
            }
            for (int64_t f = f0; f < f1;) {
                int64_t r = f / S, hi = min64(f1, (r + 1) * S);
                int64_t x = x0 + (f - f0), po = f - r * S, len = hi - f;
                if (have && pr == r && px + pn == x && pp + pn == po) {
                    pn += len;
                } else {
                    if (have) {
                        if (run) { int64_t *q = run + 5 * nr; q[0] = b; q[1] = pr; q[2] = px; q[3] = pp; q[4] = pn; }
                        ++nr;
                    }
                    have = 1; pr = r; px = x; pp = po; pn = len;
                }
                f = hi;
            }
        }
        if (have) {
            if (run) { int64_t *q = run + 5 * nr; q[0] = b; q[1] = pr; q[2] = px; q[3] = pp; q[4] = pn; }
            ++nr;
        }
    }

    if (offset) memcpy(offset, o, (size_t)n * sizeof(int64_t));
    if (bucket_of) memcpy(bucket_of, bof, (size_t)n * sizeof(int64_t));
    if (bucket_pos) memcpy(bucket_pos, pos, (size_t)n * sizeof(int64_t));
    if (dims) { dims[0] = T; dims[1] = P; dims[2] = S; dims[3] = nb; dims[4] = ns; dims[5] = nr; }
    free(o); free(bof); free(pos); free(seen);
    return ZRO_OK;
}

/*
 * The flat index of every position of bucket b under an arrival order: param
 * i's element e sits at bucket position bucket_pos[i] + e and is flat element
 * o_i + e; padding position pad_pos + j is flat element T + j.
 */
int zro_bucket_flat_map(const int64_t *numel, int64_t n, const int64_t *bucket_of, const int64_t *bucket_pos,
                        int64_t b, int64_t T, int64_t pad_pos, int64_t P, int64_t *flat_of)
{
    if (n < 0) return ZRO_EINVAL;
    int64_t o = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (bucket_of[i] == b)
            for (int64_t e = 0; e < numel[i]; ++e) flat_of[bucket_pos[i] + e] = o + e;
        o += numel[i];
    }
    if (pad_pos >= 0)
        for (int64_t j = 0; j < P - T; ++j) flat_of[pad_pos + j] = T + j;
    return ZRO_OK;
}

/* ------------------------------------------------------------------------- */
/* IPG bucket packing                                                          */
/* ------------------------------------------------------------------------- */

/*
 * Copies every replica's per-parameter grads of one bucket into that
 * replica's dense bucket buffer: element e of param i lands at bucket offset
 * o_i - bucket_start + e. Bucket positions past T (the tail padding) are set
 * to zero. ([DS] §四: each param's grad is copied into the contiguous
 * reduce_bucket_size bucket as soon as it is produced; §五 contiguous_gradients.)
 *
 * grads[k * n + i] is replica k's grad of param i (only params of this
 * bucket are read); out[k] receives numel_b = bucket_end - bucket_start
 * elements. elem_size is 2 (bf16) or 4 (fp32): packing moves bits only.
 */
int zro_bucket_pack(const int64_t *numel, const int64_t *offset, int64_t n, int32_t world,
                    int64_t T, int64_t bucket_start, int64_t bucket_end,
                    const void *const *grads, int32_t elem_size, void *const *out)
{
    if (world < 1 || (elem_size != 2 && elem_size != 4) || bucket_end < bucket_start) return ZRO_EINVAL;
    for (int32_t k = 0; k < world; ++k) {
        unsigned char *dst = (unsigned char *)out[k];
        for (int64_t i = 0; i < n; ++i) {
            if (offset[i] < bucket_start || offset[i] >= bucket_end) continue;
            const unsigned char *src = (const unsigned char *)grads[(int64_t)k * n + i];
            for (int64_t e = 0; e < numel[i]; ++e)
                for (int32_t c = 0; c < elem_size; ++c)
                    dst[(offset[i] - bucket_start + e) * elem_size + c] = src[e * elem_size + c];
        }
        for (int64_t f = (T > bucket_start ? T : bucket_start); f < bucket_end; ++f)
            for (int32_t c = 0; c < elem_size; ++c)
                dst[(f - bucket_start) * elem_size + c] = 0;
    }
    return ZRO_OK;
}

/*
 * The same packing under an arrival order: param i of bucket b lands at its
 * bucket position bucket_pos[i]; the padding positions [pad_pos, pad_pos +
 * P - T) of the bucket that holds them are zeroed (pad_pos < 0: none).
 */
int zro_bucket_pack_ordered(const int64_t *numel, int64_t n, int32_t world, const int64_t *bucket_of,
                            const int64_t *bucket_pos, int64_t b, int64_t pad_pos, int64_t pad_n,
                            const void *const *grads, int32_t elem_size, void *const *out)
{
    if (world < 1 || (elem_size != 2 && elem_size != 4) || pad_n < 0) return ZRO_EINVAL;
    for (int32_t k = 0; k < world; ++k) {
        unsigned char *dst = (unsigned char *)out[k];
        for (int64_t i = 0; i < n; ++i) {
            if (bucket_of[i] != b) continue;
            const unsigned char *src = (const unsigned char *)grads[(int64_t)k * n + i];
            for (int64_t e = 0; e < numel[i]; ++e)
                for (int32_t c = 0; c < elem_size; ++c)
                    dst[(bucket_pos[i] + e) * elem_size + c] = src[e * elem_size + c];
        }
        if (pad_pos >= 0)
            for (int64_t j = 0; j < pad_n; ++j)
                for (int32_t c = 0; c < elem_size; ++c) dst[(pad_pos + j) * elem_size + c] = 0;
    }
    return ZRO_OK;
}

/* ------------------------------------------------------------------------- */
/* Averaging: reduce-scatter and all-reduce with 1/N predivide                 */
/* ------------------------------------------------------------------------- */

/*
 * The averaged gradient of one element: each replica's value is widened to
 * fp32, multiplied by the predivide factor s (1/N, or dp/sp's reciprocal),
 * and the products are summed in fp32 in rank order 0..N-1 starting from 0
 * ([DS] §六 mean semantics: divide by dp_world_size before the reduction so
 * the sum is the mean; [MG] §"四步接力": grad_data *= 1/DP turns the sum into
 * the mean; [IQ] §"三种原语": the reduction is an element-wise sum).
 */
static float average_one(int32_t world, const void *const *x, int32_t dtype, int64_t i, float s)
{
    float acc = 0.0f;
    for (int32_t k = 0; k < world; ++k) {
        float t = load_elem(x[k], dtype, i) * s;
        acc = acc + t;
    }
    return acc;
}

/*
 * Reduce-scatter with average over one bucket: for every flat position f in
 * [bucket_start, bucket_start + numel_b), rank r = f / S receives the averaged
 * gradient at offset f - rS of its partition buffer shard[r]
 * ([IQ] §"三种原语": GPU i obtains segment i of the sum; [MG] §"通信模式":
 * each card gets only the summed gradient of its own slice; [DS] §三.3:
 * copy_grads_in_partition places the reduced slice in the local contiguous
 * partition buffer).
 * x[k] is replica k's bucket (numel_b elements of dtype).
 */
int zro_reduce_scatter_avg(int32_t world, int64_t S, int64_t bucket_start, int64_t numel_b,
                           const void *const *x, int32_t dtype, float s, float *const *shard)
{
    if (world < 1 || S < 1 || numel_b < 0) return ZRO_EINVAL;
    for (int64_t e = 0; e < numel_b; ++e) {
        int64_t f = bucket_start + e;
        int64_t r = f / S;
        shard[r][f - r * S] = average_one(world, x, dtype, e, s);
    }
    return ZRO_OK;
}

/* The same for a bucket whose position e holds flat element flat_of[e]
 * (an arrival order other than the flat one). */
int zro_reduce_scatter_avg_map(int32_t world, int64_t S, int64_t numel_b, const int64_t *flat_of,
                               const void *const *x, int32_t dtype, float s, float *const *shard)
{
    if (world < 1 || S < 1 || numel_b < 0) return ZRO_EINVAL;
    for (int64_t e = 0; e < numel_b; ++e) {
        int64_t f = flat_of[e];
        int64_t r = f / S;
        shard[r][f - r * S] = average_one(world, x, dtype, e, s);
    }
    return ZRO_OK;
}

/*
 * All-reduce with average over one bucket, the path taken when reduce_scatter
 * is off ([DS] §三.2, gradient_reduction_w_predivide over the whole bucket;
 * [IQ] §"三种原语": every GPU ends with the same full result): every replica k
 * receives the full averaged bucket in out[k], summed in the same order as
 * the reduce-scatter, then multiplied by `postscale`. That path keeps the
 * pre- and post-scaling of fp16 training ([DS] §三.2 gradient_predivide_factor
 * and postscale_gradients; §六: divide before the reduction, scale after):
 * with predivide factor f, s = 1/f and postscale = f/N; f = N gives
 * postscale 1, and a product by 1 is exact.
 */
int zro_allreduce_avg(int32_t world, int64_t numel_b, const void *const *x, int32_t dtype,
                      float s, float postscale, float *const *out)
{
    if (world < 1 || numel_b < 0) return ZRO_EINVAL;
    for (int64_t e = 0; e < numel_b; ++e) {
        float a = average_one(world, x, dtype, e, s) * postscale;
        for (int32_t k = 0; k < world; ++k) out[k][e] = a;
    }
    return ZRO_OK;
}

/* ------------------------------------------------------------------------- */
/* fp32 main-grad accumulation                                                 */
/* ------------------------------------------------------------------------- */

/* main_grad[e] += float(g[e]) in fp32 ([MG] §"四步接力" step 2:
 * param.main_grad.add_(param.grad) into the fp32 contiguous buffer, fp32
 * because repeated bf16 accumulation loses precision). */
int zro_grad_accumulate(int64_t n, float *main_grad, const void *g, int32_t dtype)
{
    if (n < 0) return ZRO_EINVAL;
    for (int64_t e = 0; e < n; ++e) main_grad[e] = main_grad[e] + load_elem(g, dtype, e);
    return ZRO_OK;
}

/* ------------------------------------------------------------------------- */
/* AdamW on one fp32 shard                                                     */
/* ------------------------------------------------------------------------- */

/*
 * The scalars of one AdamW step, computed in double from the fp32
 * hyper-parameters and rounded once each to fp32:
 *   out = {beta1, 1-beta1, beta2, 1-beta2, lr/(1-beta1^t), sqrt(1-beta2^t), 1-lr*wd, eps}.
 * The pages fix no optimizer formula beyond "update this card's 1/DP params
 * with the fp32 master" ([MG] §"通信模式"); this is decoupled-weight-decay
 * Adam with bias correction, as in Loshchilov & Hutter's AdamW.
 */
int zro_adamw_scalars(float lr, float beta1, float beta2, float eps, float weight_decay,
                      int64_t step, float *out)
{
    if (step < 1) return ZRO_EINVAL;
    double b1 = beta1, b2 = beta2, t = (double)step;
    double bc1 = 1.0 - pow(b1, t);
    double bc2 = 1.0 - pow(b2, t);
    out[0] = beta1;
    out[1] = (float)(1.0 - b1);
    out[2] = beta2;
    out[3] = (float)(1.0 - b2);
    out[4] = (float)((double)lr / bc1);
    out[5] = (float)sqrt(bc2);
    out[6] = (float)(1.0 - (double)lr * (double)weight_decay);
    out[7] = eps;
    return ZRO_OK;
}

/*
 * One AdamW step over n shard elements, in place, each operation rounded to
 * fp32 in the order written:
 *   m' = b1*m + (1-b1)*g
 *   v' = b2*v + (1-b2)*(g*g)
 *   d  = sqrt(v') / sqrt(1-b2^t) + eps
 *   p' = p*(1-lr*wd) - (lr/(1-b1^t)) * (m'/d)
 * ([MG] §"朴素 DP 的致命浪费": fp32 master, momentum m and variance v are the
 * 12 optimizer bytes per param; §"通信模式": each card updates its own 1/DP
 * slice with the fp32 master.)
 */
static void adamw_one(const float *c, float *p, float *m, float *v, float g)
{
    float m1 = c[0] * *m + c[1] * g;
    float gg = g * g;
    float v1 = c[2] * *v + c[3] * gg;
    float d = sqrtf(v1) / c[5] + c[7];
    float u = m1 / d;
    float p1 = *p * c[6] - c[4] * u;
    *m = m1;
    *v = v1;
    *p = p1;
}

int zro_adamw(int64_t n, float *p, float *m, float *v, const float *g,
              float lr, float beta1, float beta2, float eps, float weight_decay, int64_t step)
{
    float c[8];
    if (n < 0 || zro_adamw_scalars(lr, beta1, beta2, eps, weight_decay, step, c)) return ZRO_EINVAL;
    for (int64_t e = 0; e < n; ++e) adamw_one(c, &p[e], &m[e], &v[e], g[e]);
    return ZRO_OK;
}

/* ------------------------------------------------------------------------- */
/* All-gather payload: cast of the updated shards into the full bf16 params    */
/* ------------------------------------------------------------------------- */

/*
 * out[f] = bf16(master[f / S][f % S]) for f < T and 0 for the tail padding
 * T <= f < P ([MG] §"通信模式": all-gather concatenates every card's updated
 * slice back into the full weights for the next forward; [IQ] §"三种原语":
 * every GPU ends holding the complete data).
 */
int zro_gather_cast_bf16(int32_t world, int64_t T, int64_t S, const float *const *master,
                         uint16_t *out)
{
    if (world < 1 || S < 0) return ZRO_EINVAL;
    int64_t P = S * world;
    for (int64_t f = 0; f < P; ++f) {
        int64_t r = f / S;
        out[f] = f < T ? f32_to_bf16(master[r][f - r * S]) : (uint16_t)0;
    }
    return ZRO_OK;
}

/*
 * The whole step for one bucket, composed from the pieces above in the
 * pages' order ([MG] §"通信模式": reduce-scatter, then the fp32 update of the
 * local slice, then the all-gather of the updated params):
 *   1. average the bucket into a scratch fp32 array and place it by partition;
 *   2. AdamW on every partition slice the bucket covers;
 *   3. bf16 cast of those updated master elements into param_bf16 (flat index),
 *      zero for the padding.
 * grad_out (may be NULL) receives the averaged gradient by partition, as the
 * reduce-scatter would. param_bf16 may be NULL.
 */
int zro_rs_adam_fused(int32_t world, int64_t T, int64_t S, int64_t bucket_start, int64_t numel_b,
                      const void *const *x, int32_t dtype, float s,
                      float *const *master, float *const *m, float *const *v,
                      float lr, float beta1, float beta2, float eps, float weight_decay, int64_t step,
                      uint16_t *param_bf16, float *const *grad_out)
{
    float c[8];
    if (world < 1 || S < 1 || numel_b < 0) return ZRO_EINVAL;
    if (zro_adamw_scalars(lr, beta1, beta2, eps, weight_decay, step, c)) return ZRO_EINVAL;
    float *avg = (float *)malloc((size_t)(numel_b > 0 ? numel_b : 1) * sizeof(float));
    if (!avg) return -3;
    for (int64_t e = 0; e < numel_b; ++e) avg[e] = average_one(world, x, dtype, e, s);
    for (int64_t e = 0; e < numel_b; ++e) {
        int64_t f = bucket_start + e;
        int64_t r = f / S, j = f - r * S;
        if (grad_out) grad_out[r][j] = avg[e];
        adamw_one(c, &master[r][j], &m[r][j], &v[r][j], avg[e]);
        if (param_bf16) param_bf16[f] = f < T ? f32_to_bf16(master[r][j]) : (uint16_t)0;
    }
    free(avg);
    return ZRO_OK;
}

/* The same for a bucket whose position e holds flat element flat_of[e]. */
int zro_rs_adam_fused_map(int32_t world, int64_t T, int64_t S, int64_t numel_b, const int64_t *flat_of,
                          const void *const *x, int32_t dtype, float s,
                          float *const *master, float *const *m, float *const *v,
                          float lr, float beta1, float beta2, float eps, float weight_decay, int64_t step,
                          uint16_t *param_bf16, float *const *grad_out)
{
    float c[8];
    if (world < 1 || S < 1 || numel_b < 0) return ZRO_EINVAL;
    if (zro_adamw_scalars(lr, beta1, beta2, eps, weight_decay, step, c)) return ZRO_EINVAL;
    for (int64_t e = 0; e < numel_b; ++e) {
        float a = average_one(world, x, dtype, e, s);
        int64_t f = flat_of[e];
        int64_t r = f / S, j = f - r * S;
        if (grad_out) grad_out[r][j] = a;
        adamw_one(c, &master[r][j], &m[r][j], &v[r][j], a);
        if (param_bf16) param_bf16[f] = f < T ? f32_to_bf16(master[r][j]) : (uint16_t)0;
    }
    return ZRO_OK;
}

/* ------------------------------------------------------------------------- */
/* Global gradient check before the step, and the step it steers               */
/* ------------------------------------------------------------------------- */

/*
 * Runs once every bucket has been averaged into the partitions and before
 * the optimizer step ([MG] §"跨 model-parallel 的梯度收尾": DP sync first,
 * then the remaining gradient fix-ups, then optimizer.step(); [DS] §六: fp16
 * training guards the gradient arithmetic). The pages give no formula, so
 * this is the usual one:
 *   sumsq     = sum over r = 0..N-1, j = 0..S-1 (flat order) of g[r][j]^2,
 *               each square exact in double (a 24-bit significand squared
 *               fits in 53 bits), summed in double;
 *   norm      = sqrt(sumsq), in double (the global L2 norm of the averaged
 *               gradient over every rank's partition);
 *   nonfinite = the number of elements whose fp32 square g*g is not finite
 *               (NaN, an infinity, or |g| so large that its square
 *               overflows fp32);
 *   skip      = nonfinite > 0: the step changes nothing (an overflowed
 *               step is dropped, as fp16 loss scaling does);
 *   coef      = fp32(min(1, max_norm / (norm + 1e-6))), computed in double
 *               and rounded once, when max_norm > 0 and skip == 0; else 1
 *               (gradient clipping by the global norm).
 * g[r] is rank r's averaged shard gradient (S fp32).
 */
int zro_grad_check(int32_t world, int64_t S, const float *const *g, float max_norm,
                   double *sumsq, int64_t *nonfinite, double *norm, float *coef, int32_t *skip)
{
    if (world < 1 || S < 0) return ZRO_EINVAL;
    double acc = 0.0;
    int64_t bad = 0;
    for (int32_t r = 0; r < world; ++r)
        for (int64_t j = 0; j < S; ++j) {
            float x = g[r][j];
            float sq32 = x * x;
            if (!isfinite(sq32)) ++bad;
            double d = (double)x;
            acc = acc + d * d;
        }
    double nrm = sqrt(acc);
    float c = 1.0f;
    if (max_norm > 0.0f && bad == 0) {
        double q = (double)max_norm / (nrm + 1e-6);
        c = q < 1.0 ? (float)q : 1.0f;
    }
    *sumsq = acc;
    *nonfinite = bad;
    *norm = nrm;
    *coef = c;
    *skip = bad > 0;
    return ZRO_OK;
}

/*
 * The step the check steers, over every rank's shard: if skip, nothing is
 * written. Otherwise, for every rank r and shard element j:
 *   gc = g[r][j] * coef (fp32, rounded; exact when coef = 1),
 *   AdamW on master[r][j], m[r][j], v[r][j] with gc (adamw_one above),
 *   param_bf16[rS + j] = bf16(master[r][j]) for rS + j < T, 0 for the padding
 * ([MG] §"通信模式": the fp32 update of the local slice, then the
 * all-gather's payload). param_bf16 may be NULL.
 */
int zro_adam_clip_step(int32_t world, int64_t T, int64_t S, float *const *master, float *const *m,
                       float *const *v, const float *const *g, float coef, int32_t skip,
                       float lr, float beta1, float beta2, float eps, float weight_decay, int64_t step,
                       uint16_t *param_bf16)
{
    float c[8];
    if (world < 1 || S < 0) return ZRO_EINVAL;
    if (zro_adamw_scalars(lr, beta1, beta2, eps, weight_decay, step, c)) return ZRO_EINVAL;
    if (skip) return ZRO_OK;
    for (int32_t r = 0; r < world; ++r)
        for (int64_t j = 0; j < S; ++j) {
            float gc = g[r][j] * coef;
            adamw_one(c, &master[r][j], &m[r][j], &v[r][j], gc);
            if (param_bf16) {
                int64_t f = (int64_t)r * S + j;
                param_bf16[f] = f < T ? f32_to_bf16(master[r][j]) : (uint16_t)0;
            }
        }
    return ZRO_OK;
}

/* ------------------------------------------------------------------------- */
/* Byte accounting                                                             */
/* ------------------------------------------------------------------------- */

/*
 * Bytes one rank sends (= receives) per step for gradient averaging and the
 * parameter refresh, over the padded flat buffer of P = N*S elements of
 * elem_bytes each, counting ring collectives ([MG] §"NCCL 底层算法": ring
 * all-reduce moves 2(N-1)/N of the message per card, half in its
 * reduce-scatter phase and half in its all-gather phase; [IQ] §"Ring=RS+AG"):
 *   scheme 0: DP all-reduce of the grads                 2(N-1) S e
 *   scheme 1: first ZeRO-1, all-reduce + param all-gather 3(N-1) S e   (1.5x of DP)
 *   scheme 2: partition-aware reduce-scatter + all-gather 2(N-1) S e   (1.0x of DP)
 *   scheme 3: reduce-scatter alone                        (N-1) S e    (the gradient half)
 * ([DS] §一: total communication cut from 1.5x to 1.0x of data parallelism.)
 */
int zro_comm_bytes(int32_t scheme, int32_t world, int64_t S, int32_t elem_bytes, double *out)
{
    if (world < 1 || S < 0 || elem_bytes < 1) return ZRO_EINVAL;
    double unit = (double)(world - 1) * (double)S * (double)elem_bytes;
    switch (scheme) {
    case 0: *out = 2.0 * unit; break;
    case 1: *out = 3.0 * unit; break;
    case 2: *out = 2.0 * unit; break;
    case 3: *out = 1.0 * unit; break;
    default: return ZRO_EINVAL;
    }
    return ZRO_OK;
}

/*
 * Per-rank memory for weights, grads and optimizer state, mixed precision
 * with Adam ([MG] §"朴素 DP 的致命浪费": bf16 weight 2 + bf16 grad 2 + fp32
 * master 4 + m 4 + v 4 = 16 bytes per param; §"ZeRO 各档" table): unsharded
 * items cover all T params, sharded ones the S elements of one partition.
 *   stage 0  (plain DP):   16 T
 *   stage 1  (ZeRO-1):     2 T + 2 T + 12 S
 *   stage 15 (ZeRO-1.5/2): 2 T + 2 S + 12 S
 *   stage 3  (ZeRO-3):     16 S
 */
int zro_layout_bytes(int32_t stage, int64_t T, int64_t S, double *out)
{
    if (T < 0 || S < 0) return ZRO_EINVAL;
    double t = (double)T, s = (double)S;
    switch (stage) {
    case 0: *out = 16.0 * t; break;
    case 1: *out = 2.0 * t + 2.0 * t + 12.0 * s; break;
    case 15: *out = 2.0 * t + 2.0 * s + 12.0 * s; break;
    case 3: *out = 16.0 * s; break;
    default: return ZRO_EINVAL;
    }
    return ZRO_OK;
}

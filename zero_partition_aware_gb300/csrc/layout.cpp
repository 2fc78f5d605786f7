// layout.cpp -- host-only part of libzr's C ABI: status and error messages,
// the flat partitioned layout with its buckets, slices and runs, the AdamW
// scalar preparation and the byte accounting.
//
// Sources, cited by page title and section:
//   [DS] "DeepSpeed ZeRO 通信优化深度解析：用 reduce-scatter 分区感知规约替代 all-reduce"
//   [MG] "Megatron-LM 分布式训练（四）：数据并行 DP 与分布式优化器（ZeRO）"
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>

#include "zr_internal.h"

namespace zr {

static thread_local std::string g_last_error;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = std::string(zr_status_string(code)) + ": " + buf;
    return code;
}

void clear_error() { g_last_error.clear(); }

int prepare_adamw(const zr_adamw *hp, zr_adamw_scalars *out) {
    if (!hp || !out) return fail(ZR_ERR_INVALID_ARG, "NULL AdamW hyper-parameters");
    if (hp->step < 1) return fail(ZR_ERR_INVALID_ARG, "AdamW step %lld < 1", (long long)hp->step);
    const float vals[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
    for (float x : vals)
        if (!std::isfinite(x)) return fail(ZR_ERR_INVALID_ARG, "non-finite AdamW hyper-parameter");
    if (!(hp->beta1 >= 0.f && hp->beta1 < 1.f) || !(hp->beta2 >= 0.f && hp->beta2 < 1.f))
        return fail(ZR_ERR_INVALID_ARG, "AdamW betas must lie in [0, 1)");
    if (!(hp->eps > 0.f)) return fail(ZR_ERR_INVALID_ARG, "AdamW eps must be > 0");
    // Bias corrections in double from the fp32 inputs, each result rounded once.
    const double b1 = hp->beta1, b2 = hp->beta2, t = (double)hp->step;
    const double one_minus_b1t = 1.0 - std::pow(b1, t);
    const double one_minus_b2t = 1.0 - std::pow(b2, t);
    out->beta1 = hp->beta1;
    out->one_minus_beta1 = (float)(1.0 - b1);
    out->beta2 = hp->beta2;
    out->one_minus_beta2 = (float)(1.0 - b2);
    out->step_size = (float)((double)hp->lr / one_minus_b1t);
    out->bc2_sqrt = (float)std::sqrt(one_minus_b2t);
    out->decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
    out->eps = hp->eps;
    if (!(out->bc2_sqrt > 0.f) || !std::isfinite(out->step_size))
        return fail(ZR_ERR_INVALID_ARG, "AdamW bias correction underflows at this step");
    return ZR_OK;
}

}  // namespace zr

using zr::fail;

extern "C" {

const char *zr_status_string(int status) {
    switch (status) {
        case ZR_OK: return "ZR_OK";
        case ZR_ERR_INVALID_ARG: return "ZR_ERR_INVALID_ARG";
        case ZR_ERR_CUDA: return "ZR_ERR_CUDA";
        case ZR_ERR_OOM: return "ZR_ERR_OOM";
        case ZR_ERR_ALIGN: return "ZR_ERR_ALIGN";
        case ZR_ERR_TIMEOUT: return "ZR_ERR_TIMEOUT";
        case ZR_ERR_STATE: return "ZR_ERR_STATE";
        case ZR_ERR_UNSUPPORTED: return "ZR_ERR_UNSUPPORTED";
        default: return "ZR_ERR_UNKNOWN";
    }
}

int zr_last_error(char *buf, size_t cap) {
    const std::string &m = zr::g_last_error;
    if (buf && cap > 0) {
        size_t k = m.size() < cap - 1 ? m.size() : cap - 1;
        memcpy(buf, m.data(), k);
        buf[k] = '\0';
    }
    return (int)m.size();
}

int zr_version(void) { return 1; }

// ---------------------------------------------------------------------------
// Layout
// ---------------------------------------------------------------------------

// The flat layout ([DS] §二, [MG] §"分布式优化器"), its buckets ([DS] §四/§五),
// per-param slices ([DS] §三.2) and per-bucket runs. The buckets fill in the
// order the grads arrive (the flat order unless `arrival` says otherwise:
// backward produces the last layers first, and each grad is copied into the
// IPG bucket as soon as it is produced, [DS] §四); the flat layout and the
// partitions do not depend on it. A run is a maximal stretch of a bucket that
// is also one stretch of one partition: walking the bucket in bucket order,
// a param's piece (or the padding's) joins the previous one when it continues
// it both in the bucket and in the partition ([DS] §三.2, merging a bucket's
// same-destination fragments). In flat order the runs are the bucket x
// partition intersections.
int zr_layout_create_ordered(const int64_t *numel, int64_t n_params, int32_t world,
                             int64_t reduce_bucket_size, const int64_t *arrival, zr_layout **out) {
    zr::clear_error();
    if (!out) return fail(ZR_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (n_params < 0) return fail(ZR_ERR_INVALID_ARG, "n_params %lld < 0", (long long)n_params);
    if (n_params > 0 && !numel) return fail(ZR_ERR_INVALID_ARG, "numel is NULL");
    if (world < 1 || world > ZR_MAX_WORLD)
        return fail(ZR_ERR_INVALID_ARG, "world %d outside [1, %d]", world, ZR_MAX_WORLD);
    if (reduce_bucket_size < 1)
        return fail(ZR_ERR_INVALID_ARG, "reduce_bucket_size %lld < 1", (long long)reduce_bucket_size);
    const int64_t kMaxTotal = (int64_t)1 << 50;  // keeps every index product inside int64
    int64_t T = 0;
    for (int64_t i = 0; i < n_params; ++i) {
        if (numel[i] < 1)
            return fail(ZR_ERR_INVALID_ARG, "numel[%lld] = %lld < 1", (long long)i, (long long)numel[i]);
        if (numel[i] > kMaxTotal - T) return fail(ZR_ERR_UNSUPPORTED, "total element count above 2^50");
        T += numel[i];
    }

    zr_layout *L = new (std::nothrow) zr_layout();
    if (!L) return fail(ZR_ERR_OOM, "layout handle");
    try {
        L->arrival.resize(n_params);
        if (arrival) {
            std::vector<char> seen(n_params, 0);
            for (int64_t k = 0; k < n_params; ++k) {
                const int64_t i = arrival[k];
                if (i < 0 || i >= n_params || seen[i]) {
                    delete L;
                    return fail(ZR_ERR_INVALID_ARG, "arrival is not a permutation of the params (entry %lld)",
                                (long long)k);
                }
                seen[i] = 1;
                L->arrival[k] = i;
            }
        } else {
            for (int64_t k = 0; k < n_params; ++k) L->arrival[k] = k;
        }
        L->world = world;
        L->bucket_size = reduce_bucket_size;
        L->T = T;
        L->P = (T + world - 1) / world * world;
        L->S = L->P / world;
        const int64_t S = L->S;
        L->numel.assign(numel, numel + n_params);
        L->offset.resize(n_params);
        L->bucket_of.resize(n_params);
        L->bucket_pos.resize(n_params);
        for (int64_t i = 0, o = 0; i < n_params; ++i) {
            L->offset[i] = o;
            o += numel[i];
        }
        // buckets: consecutive stretches of the arrival order, closed before an overflow
        for (int64_t k = 0; k < n_params;) {
            int64_t j = k, fill = 0;
            const int64_t b = L->n_buckets();
            while (j < n_params && (fill == 0 || fill + numel[L->arrival[j]] <= reduce_bucket_size)) {
                const int64_t i = L->arrival[j];
                L->bucket_of[i] = b;
                L->bucket_pos[i] = fill;
                fill += numel[i];
                ++j;
            }
            bool in_order = true;
            for (int64_t q = k + 1; q < j; ++q) in_order = in_order && L->arrival[q] == L->arrival[q - 1] + 1;
            L->b_arr_lo.push_back(k);
            L->b_arr_hi.push_back(j);
            L->b_size.push_back(fill);
            L->b_pad_pos.push_back(-1);
            L->b_flat_start.push_back(in_order ? L->offset[L->arrival[k]] : -1);
            k = j;
        }
        if (n_params > 0) {  // the padding travels with the bucket of the last flat param
            const int64_t pb = L->bucket_of[n_params - 1];
            L->b_pad_pos[pb] = L->b_size[pb];
            L->b_size[pb] += L->P - T;
            if (L->arrival[L->b_arr_hi[pb] - 1] != n_params - 1) L->b_flat_start[pb] = -1;
        }
        // runs, bucket by bucket in bucket order
        for (int64_t b = 0; b < L->n_buckets(); ++b) {
            L->b_run_lo.push_back((int64_t)L->runs.size());
            bool open = false;
            zr_run cur{};
            auto piece = [&](int64_t f0, int64_t f1, int64_t x0) {
                for (int64_t f = f0; f < f1;) {
                    const int64_t r = f / S, hi = f1 < (r + 1) * S ? f1 : (r + 1) * S;
                    const int64_t x = x0 + (f - f0), po = f - r * S, n = hi - f;
                    if (open && cur.dst == r && cur.bucket_offset + cur.numel == x &&
                        cur.partition_offset + cur.numel == po) {
                        cur.numel += n;
                    } else {
                        if (open) L->runs.push_back(cur);
                        cur = zr_run{};
                        cur.bucket = b;
                        cur.dst = (int32_t)r;
                        cur.bucket_offset = x;
                        cur.partition_offset = po;
                        cur.numel = n;
                        open = true;
                    }
                    f = hi;
                }
            };
            for (int64_t k = L->b_arr_lo[b]; k < L->b_arr_hi[b]; ++k) {
                const int64_t i = L->arrival[k];
                piece(L->offset[i], L->offset[i] + numel[i], L->bucket_pos[i]);
            }
            if (L->b_pad_pos[b] >= 0) piece(T, L->P, L->b_pad_pos[b]);
            if (open) L->runs.push_back(cur);
            L->b_run_hi.push_back((int64_t)L->runs.size());
        }
        // slices: param x partition intersections
        L->p_slice_lo.resize(n_params + 1);
        for (int64_t p = 0; p < n_params; ++p) {
            L->p_slice_lo[p] = (int64_t)L->slices.size();
            const int64_t o = L->offset[p], n = numel[p];
            for (int64_t r = o / S; r * S < o + n; ++r) {
                const int64_t lo = o > r * S ? o : r * S;
                const int64_t hi = o + n < (r + 1) * S ? o + n : (r + 1) * S;
                zr_slice sl{};
                sl.param = p;
                sl.bucket = L->bucket_of[p];
                sl.dst = (int32_t)r;
                sl.param_offset = lo - o;
                sl.bucket_offset = L->bucket_pos[p] + lo - o;
                sl.partition_offset = lo - r * S;
                sl.numel = hi - lo;
                L->slices.push_back(sl);
            }
        }
        L->p_slice_lo[n_params] = (int64_t)L->slices.size();
    } catch (const std::bad_alloc &) {
        delete L;
        return fail(ZR_ERR_OOM, "layout tables");
    }
    *out = L;
    return ZR_OK;
}

int zr_layout_create(const int64_t *numel, int64_t n_params, int32_t world,
                     int64_t reduce_bucket_size, zr_layout **out) {
    return zr_layout_create_ordered(numel, n_params, world, reduce_bucket_size, nullptr, out);
}

int zr_layout_destroy(zr_layout *layout) {
    delete layout;
    return ZR_OK;
}

int zr_layout_query(const zr_layout *L, zr_layout_info *info) {
    zr::clear_error();
    if (!L || !info) return fail(ZR_ERR_INVALID_ARG, "NULL argument");
    info->T = L->T;
    info->P = L->P;
    info->S = L->S;
    info->n_params = L->n_params();
    info->n_buckets = L->n_buckets();
    info->n_slices = (int64_t)L->slices.size();
    info->n_runs = (int64_t)L->runs.size();
    info->reduce_bucket_size = L->bucket_size;
    info->world = L->world;
    return ZR_OK;
}

int zr_layout_param_partitions(const zr_layout *L, int64_t param, int32_t *part_ids,
                               int64_t *grad_start_offset, int32_t cap, int32_t *n_out) {
    zr::clear_error();
    if (!L || !n_out) return fail(ZR_ERR_INVALID_ARG, "NULL argument");
    if (param < 0 || param >= L->n_params())
        return fail(ZR_ERR_INVALID_ARG, "param %lld out of range", (long long)param);
    const int64_t lo = L->p_slice_lo[param], hi = L->p_slice_lo[param + 1];
    *n_out = (int32_t)(hi - lo);
    for (int64_t k = lo; k < hi && k - lo < cap; ++k) {
        if (part_ids) part_ids[k - lo] = L->slices[k].dst;
        if (grad_start_offset) grad_start_offset[k - lo] = L->slices[k].param_offset;
    }
    return ZR_OK;
}

int zr_layout_slices(const zr_layout *L, zr_slice *out, int64_t cap, int64_t *n_out) {
    zr::clear_error();
    if (!L || !n_out) return fail(ZR_ERR_INVALID_ARG, "NULL argument");
    *n_out = (int64_t)L->slices.size();
    if (out)
        for (int64_t k = 0; k < *n_out && k < cap; ++k) out[k] = L->slices[k];
    return ZR_OK;
}

int zr_layout_runs(const zr_layout *L, zr_run *out, int64_t cap, int64_t *n_out) {
    zr::clear_error();
    if (!L || !n_out) return fail(ZR_ERR_INVALID_ARG, "NULL argument");
    *n_out = (int64_t)L->runs.size();
    if (out)
        for (int64_t k = 0; k < *n_out && k < cap; ++k) out[k] = L->runs[k];
    return ZR_OK;
}

int zr_layout_bucket(const zr_layout *L, int64_t b, int64_t *flat_start, int64_t *numel) {
    zr::clear_error();
    if (!L) return fail(ZR_ERR_INVALID_ARG, "NULL layout");
    if (b < 0 || b >= L->n_buckets()) return fail(ZR_ERR_INVALID_ARG, "bucket %lld out of range", (long long)b);
    if (flat_start) *flat_start = L->b_flat_start[b];
    if (numel) *numel = L->b_size[b];
    return ZR_OK;
}

int zr_layout_param(const zr_layout *L, int64_t param, int64_t *flat_offset, int64_t *bucket) {
    zr::clear_error();
    if (!L) return fail(ZR_ERR_INVALID_ARG, "NULL layout");
    if (param < 0 || param >= L->n_params())
        return fail(ZR_ERR_INVALID_ARG, "param %lld out of range", (long long)param);
    if (flat_offset) *flat_offset = L->offset[param];
    if (bucket) *bucket = L->bucket_of[param];
    return ZR_OK;
}

int zr_layout_bucket_positions(const zr_layout *L, int64_t *out, int64_t cap, int64_t *n_out) {
    zr::clear_error();
    if (!L) return fail(ZR_ERR_INVALID_ARG, "NULL layout");
    if (cap < 0) return fail(ZR_ERR_INVALID_ARG, "cap < 0");
    const int64_t n = L->n_params();
    if (out)
        for (int64_t i = 0; i < n && i < cap; ++i) out[i] = L->bucket_pos[i];
    if (n_out) *n_out = n;
    return ZR_OK;
}

// ---------------------------------------------------------------------------
// Accounting
// ---------------------------------------------------------------------------

int zr_adamw_prepare(const zr_adamw *hp, zr_adamw_scalars *out) {
    zr::clear_error();
    return zr::prepare_adamw(hp, out);
}

// Ring collectives over P = N*S elements: all-reduce moves 2(N-1)/N of the
// message per rank, its reduce-scatter and all-gather halves (N-1)/N each
// ([MG] §"NCCL 底层算法"; [DS] §一: 1.5x -> 1.0x of data parallelism).
int zr_comm_bytes(const zr_layout *L, int32_t scheme, int32_t elem_bytes, double *per_rank_bytes) {
    zr::clear_error();
    if (!L || !per_rank_bytes) return fail(ZR_ERR_INVALID_ARG, "NULL argument");
    if (elem_bytes < 1) return fail(ZR_ERR_INVALID_ARG, "elem_bytes < 1");
    const double half = (double)(L->world - 1) * (double)L->S * (double)elem_bytes;  // one RS or AG
    switch (scheme) {
        case 0: *per_rank_bytes = half + half; break;         // all-reduce = RS + AG
        case 1: *per_rank_bytes = half + half + half; break;  // all-reduce, then param all-gather
        case 2: *per_rank_bytes = half + half; break;         // reduce-scatter, then all-gather
        case 3: *per_rank_bytes = half; break;                // reduce-scatter alone
        default: return fail(ZR_ERR_INVALID_ARG, "scheme %d not in 0..3", scheme);
    }
    return ZR_OK;
}

// [MG] §"朴素 DP 的致命浪费" (2+2+4+4+4 bytes) and §"ZeRO 各档": unsharded
// items cover the T params, sharded items the S elements of one partition.
int zr_layout_bytes(const zr_layout *L, int32_t stage, double *bytes_per_rank) {
    zr::clear_error();
    if (!L || !bytes_per_rank) return fail(ZR_ERR_INVALID_ARG, "NULL argument");
    const double weights = 2, grads = 2, optim = 4 + 4 + 4;
    const double T = (double)L->T, S = (double)L->S;
    switch (stage) {
        case 0: *bytes_per_rank = (weights + grads + optim) * T; break;
        case 1: *bytes_per_rank = (weights + grads) * T + optim * S; break;
        case 15: *bytes_per_rank = weights * T + (grads + optim) * S; break;
        case 3: *bytes_per_rank = (weights + grads + optim) * S; break;
        default: return fail(ZR_ERR_INVALID_ARG, "stage %d not in {0, 1, 15, 3}", stage);
    }
    return ZR_OK;
}

}  // extern "C"

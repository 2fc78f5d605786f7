// zr_internal.h -- library-private declarations shared by the host-only part of
// the C ABI (layout.cpp: layout, status, accounting) and the device steps
// (kernels.cu).
#pragma once

#include <cstdarg>
#include <cstdint>
#include <string>
#include <vector>

#include "zr.h"

struct zr_layout {
    int32_t world = 1;
    int64_t bucket_size = 1;
    int64_t T = 0, P = 0, S = 0;
    std::vector<int64_t> numel, offset, bucket_of;
    std::vector<int64_t> arrival;     // the params in the order their grads arrive (fill the buckets)
    std::vector<int64_t> bucket_pos;  // per param: its position inside its bucket
    // per bucket: size (padding included), padding position (-1: none), flat
    // start (-1 unless the bucket is one flat range in flat order), its params
    // as the index range [b_arr_lo, b_arr_hi) of `arrival`, its runs
    std::vector<int64_t> b_size, b_pad_pos, b_flat_start, b_arr_lo, b_arr_hi, b_run_lo, b_run_hi;
    std::vector<zr_slice> slices;     // param order, then dst
    std::vector<int64_t> p_slice_lo;  // [n_params + 1] slice index range per param
    std::vector<zr_run> runs;         // bucket order, then bucket position
    int64_t n_params() const { return (int64_t)numel.size(); }
    int64_t n_buckets() const { return (int64_t)b_size.size(); }
};

namespace zr {

// Thread-local error message; returns `code` so callers can `return fail(...)`.
int fail(int code, const char *fmt, ...);
void clear_error();

// floor / ceil division for possibly negative numerators, positive divisor
inline int64_t floordiv(int64_t a, int64_t b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }
inline int64_t ceildiv(int64_t a, int64_t b) { return -floordiv(-a, b); }

// Host-side AdamW scalar preparation (double, rounded once to fp32).
int prepare_adamw(const zr_adamw *hp, zr_adamw_scalars *out);
}  // namespace zr

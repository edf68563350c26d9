// The plan object behind ebin_plan_t, shared by the translation units that
// execute plans.  Not part of the public C ABI.
#pragma once

#include <atomic>
#include <cstdint>

#include "ebin.h"
#include "ebin_launch.h"

struct ebin_plan_s {
    std::atomic<int> refs{1};
    // cache key
    uint64_t desc_id = 0;
    ebin_dtype dt = EBIN_FLOAT32;
    int rank_a = 0, rank_b = 0;
    int rank_c = -1;                       // three-input plans only (else -1)
    int64_t shape_a[ebin::kMaxRank] = {};
    int64_t shape_b[ebin::kMaxRank] = {};
    int64_t shape_c[ebin::kMaxRank] = {};
    // strided input views (ebin_plan_create_strided): element strides given for
    // A / B when they differ from the dense ones (part of the cache key)
    bool strided_a = false, strided_b = false;
    int64_t strides_a[ebin::kMaxRank] = {};
    int64_t strides_b[ebin::kMaxRank] = {};
    // what execution needs (copied: a plan may outlive its descriptor)
    int op = 0;
    ebin_attrs attrs{};
    ebin_dtype out_dt = EBIN_FLOAT32;
    ebin_dtype dt_b = EBIN_FLOAT32;        // B's type (mixed-type Pow), else dt
    int rank_out = 0;
    int64_t shape_out[ebin::kMaxRank] = {};
    int64_t numel = 0, numel_a = 0, numel_b = 0, numel_c = 0;
    int64_t span_a = 0, span_b = 0;        // storage extent of A / B in elements
    ebin::Geom g{};
    int family = ebin::FAM_EMPTY;
    int64_t plane = 0;
};

namespace ebin {
// Add one to the process-wide kernel launch count (ebin_launch_count).
void count_launch();

// The checks and launch description of a two-input execution: NULL buffers,
// the alias rule, the status word and the 16-byte alignment fallback to the
// general kernel.  `status`: the device word a validating kernel ORs its bits
// into, or nullptr for the stream's own word (allocated on first use).  On
// EBIN_OK, L is ready for launch().
ebin_status prepare_launch(const ebin_plan_s &p, const void *A, const void *B, void *out,
                           cudaStream_t s, uint32_t *status, Launch &L);
}  // namespace ebin

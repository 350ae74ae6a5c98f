// The prompt chunk size for prefill under a layer split (host only).
//
// strata PR #1441 "Prompt chunks sized for a layer split's pipeline", sections
// "Summary" and "What changed": with S pipeline stages, a prompt of n tokens
// read in chunks of C passes through S - 1 + n / C stage steps, each costing a
// fixed b plus a per token, so the total is smallest at C = sqrt(n (b/a) / (S - 1)).
// The size is then put on the 256-token grid (rounded up), kept within
// [512, cap], and evened out over the chunks it needs so that no short chunk is
// left at the end; a prompt that fits in one chunk is read whole.  "Evened out"
// is read as: with k = ceil(n / C) chunks, C becomes ceil(n / k) rounded up to
// the grid.  With b/a = 1024 on four stages this gives the page's chunks for
// its four prompts (2013 -> 1024, 3865 -> 1024, 10041 -> 2048, 28998 -> 3328).
#include <cmath>

#include "kvc_internal.h"

namespace {

constexpr int64_t kGrid = 256;
constexpr int64_t kMinChunk = 512;

int64_t up_to_grid(int64_t x) { return (x + kGrid - 1) / kGrid * kGrid; }

}  // namespace

extern "C" int kvc_pipeline_chunk(int32_t n_tokens, int32_t cap, int32_t stages, double b_over_a,
                                  int32_t *chunk) {
    if (!chunk || n_tokens <= 0 || cap <= 0 || stages <= 0 || !(b_over_a > 0.0) || !std::isfinite(b_over_a))
        return KVC_EINVAL;
    const int64_t n = n_tokens;
    if (stages == 1) {  // nothing to overlap: the largest chunk the buffers allow
        *chunk = (int32_t)(n < cap ? n : cap);
        return KVC_OK;
    }
    const double best = std::sqrt((double)n * b_over_a / (double)(stages - 1));
    if (!(best < 4.0e9)) return KVC_EINVAL;
    int64_t c = up_to_grid((int64_t)std::ceil(best));
    if (c < kMinChunk) c = kMinChunk;
    if (c > cap) c = cap;
    if (c >= n) {
        *chunk = (int32_t)n;
        return KVC_OK;
    }
    const int64_t k = (n + c - 1) / c;              // chunks the size needs
    int64_t even = up_to_grid((n + k - 1) / k);     // the same number of chunks, evened out
    if (even < kMinChunk) even = kMinChunk;
    if (even > cap) even = cap;
    *chunk = (int32_t)even;
    return KVC_OK;
}

// host.h -- host-side services of attn_api.cu shared with the other entry
// points of the library: per-device state, TMA descriptor encoding, argument
// helpers.
#pragma once

#include <cuda.h>

#include <cstddef>

namespace attn {
namespace host {

// Sets up the current device once (capability 10.3, SM count, status word,
// tensor-map encoder); ATTN_OK or the reason it cannot run the kernels.
// *device receives the device's index.
int current_device(int* sm_count, unsigned int** status_word, int* device);

// Rank-3 bf16 view [outer, S, D] of a contiguous tensor on `device`, box {64
// elements, 128 rows, 1}, 128-byte swizzle, rows past S read as zero.  Served
// from a cache of encoded maps when the same view was encoded before.
int encode_bf16_tiles(CUtensorMap* map, int device, const void* ptr, int D, int S, long long outer);
// The same view with a box of `box_rows` rows (at most 256).
int encode_bf16_box(CUtensorMap* map, int device, const void* ptr, int D, int S, long long outer,
                    int box_rows);

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb);

// Bound on every device-side wait, in nanoseconds.
unsigned long long wait_limit_ns();

}  // namespace host
}  // namespace attn

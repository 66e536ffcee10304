// fa_host.h -- host-side helpers shared by the library's translation units
// (internal; not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace fa_host {

// Facts about one device, looked up once: compute capability, SM count and the
// device addresses of the status word and the scheduler counters.
struct DeviceInfo {
    cudaError_t err;
    int cc_major, cc_minor, sm_count;
    unsigned int *status;
    unsigned int *sched;
};

// nullptr-free: err is cudaErrorInvalidDevice for an out-of-range ordinal.
DeviceInfo device_info(int dev);
bool aligned16(const void *p);
bool aligned32(const void *p);
bool aligned4(const void *p);
bool overlaps(const void *a, size_t na, const void *b, size_t nb);
bool on_device(const void *p, int dev);
// 3-D TMA map over a contiguous BH x N x d 16-bit tensor: box 64 columns x 128
// rows, 128-byte swizzle, rows past N read as zero.
bool make_map(CUtensorMap *map, const void *base, bool bf16, int64_t BH, int64_t N, int64_t d,
              uint32_t box_rows = 128);
// The same over a token-major tokens x heads x d tensor, ordered (d, heads,
// tokens) with a 64-column x 1-head x box_tokens-token box.
bool make_map_tokens(CUtensorMap *map, const void *base, bool bf16, int64_t tokens, int64_t heads,
                     int64_t d, uint32_t box_tokens = 128);
uint64_t wait_budget();
void count_launches(int64_t n);
// The armed test-hook position (fa_test_arm_fault), disarming it; -1 if none.
int take_fault_position();
// The scheduler counters of one launch (a slot of the device's static array,
// zero at launch; the launch's last CTA zeroes it again).
unsigned int *next_sched_slot(unsigned int *base);
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace fa_host

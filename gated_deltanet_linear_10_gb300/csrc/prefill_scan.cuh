// Shared declarations of the chunk-state scan (internal header): the slot
// lists scan_setup_kernel derives on the device, the scratch layout, and the
// host launchers in prefill_scan.cu.
#pragma once

#include <stdint.h>

#include <cuda_runtime.h>

#include "gdn.h"

namespace gdn {
namespace scan {

constexpr int kChunk = 64;
// scratch state slots (each hv x 128 x 128 fp32): S_1 (segment 0's final
// state), B (segment 1 from zero), A (segment 1 from the identity, v = 0)
constexpr int kSlotS1 = 0, kSlotB = 1, kSlotA = 2, kScratchSlots = 3;
constexpr uint32_t kS1bBytes = 128 * 128 * 2;      // S_1 as a bf16 operand, per head

struct ScanIdx {
    int32_t cu_all[3];      // segment bounds: [start, cut, end)
    int32_t init[2];        // initial slots of segments 0 and 1 (caller's pool)
    int32_t fin[2];         // final slots of segments 0 and 1 (scratch)
    int32_t final_slot;     // the caller's final slot (< 0: not written)
};

}  // namespace scan

gdn_status scan_setup(const int32_t *cu, int64_t n_tokens, const int32_t *ii, const int32_t *fi,
                      int64_t n_slots, scan::ScanIdx *idx, cudaStream_t s);
gdn_status scan_finish(const float *states, int hv, const scan::ScanIdx *idx, float *pool,
                       uint8_t *s1b, const void *phi, int64_t phi_rows, void *o, int64_t n_tokens,
                       cudaStream_t s);
gdn_status read_status_prefill_scan(uint32_t *out, int clear, cudaStream_t s);

}  // namespace gdn

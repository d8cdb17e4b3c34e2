// Tensor-core (tcgen05 / TMEM / TMA) chunked prefill for bf16, dk = dv = 128,
// chunk 64.  Not built yet: the generic kernel serves every shape.
#include "common.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_prefill_tc)
GDN_STATUS_READER(read_status_prefill_tc, g_status_prefill_tc)

bool prefill_tc_supported(int, int, int, int, const void *, int64_t, const void *, int64_t,
                          const void *, int64_t) {
    return false;
}

gdn_status prefill_tc(const void *, int64_t, const void *, int64_t, const void *, int64_t,
                      const float *, const float *, const int32_t *, int, int64_t, int, int,
                      float, int, float *, int64_t, const int32_t *, const int32_t *, void *,
                      cudaStream_t) {
    return GDN_ERR_UNSUPPORTED;
}

}  // namespace gdn

// Library-level entry points: status strings, version, device status word,
// and the whole-slot state snapshot copy.
#include <stdio.h>
#include <string.h>

#include "common.cuh"

namespace gdn {

GDN_DECLARE_STATUS_WORD(g_status_api)
gdn_status read_status_norm(uint32_t *out, int clear, cudaStream_t s);   // rmsnorm.cu
GDN_STATUS_READER(read_status_api, g_status_api)

static thread_local char t_last_err[256] = "";

void set_last_cuda_error(cudaError_t e) {
    snprintf(t_last_err, sizeof(t_last_err), "%s: %s", cudaGetErrorName(e),
             cudaGetErrorString(e));
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        return 1;
    return sms;
}

gdn_status launch_status() {
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return GDN_OK;
    set_last_cuda_error(e);
    return GDN_ERR_LAUNCH;
}

// Copy of whole slots, 16 bytes per thread and step.  blockIdx.y = pair.
// The "[model] support Qwen3next" review shows this operation as a buffer
// copy from source to destination indices for the MTP linear-attention
// states; here it is one kernel over all pairs.
__global__ void snapshot_kernel(uint4 *__restrict__ pool, int64_t n_slots,
                                int64_t slot_vecs, const int32_t *__restrict__ src,
                                const int32_t *__restrict__ dst) {
    griddep_wait();   // launched behind the kernel that writes the slots: nothing is read before it
    const int i = blockIdx.y;
    const int s = src[i], d = dst[i];
    if (s < 0 || d < 0) return;
    if (s >= n_slots || d >= n_slots) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag_status(GDN_DEVSTAT_BAD_INDEX);
        return;
    }
    const uint4 *from = pool + (int64_t)s * slot_vecs;
    uint4 *to = pool + (int64_t)d * slot_vecs;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    // four independent 16-byte loads in flight per thread
    for (; v + 3 * stride < slot_vecs; v += 4 * stride) {
        uint4 a = __ldcs(from + v), b = __ldcs(from + v + stride);
        uint4 c = __ldcs(from + v + 2 * stride), e = __ldcs(from + v + 3 * stride);
        __stcs(to + v, a);
        __stcs(to + v + stride, b);
        __stcs(to + v + 2 * stride, c);
        __stcs(to + v + 3 * stride, e);
    }
    for (; v < slot_vecs; v += stride) __stcs(to + v, __ldcs(from + v));
}

}  // namespace gdn

using namespace gdn;

extern "C" {

const char *gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
        case GDN_ERR_LAUNCH: return "GDN_ERR_LAUNCH";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_TOO_LARGE: return "GDN_ERR_TOO_LARGE";
    }
    return "GDN_STATUS_UNKNOWN";
}

const char *gdn_version(void) { return "gdn 0.1.0 sm_103a"; }

const char *gdn_last_cuda_error(void) { return t_last_err; }

gdn_status gdn_get_device_status(uint32_t *out, int32_t clear, void *stream) {
    GDN_REQUIRE(out != nullptr, GDN_ERR_INVALID_ARG);
    cudaStream_t s = (cudaStream_t)stream;
    *out = 0;
    gdn_status st;
    if ((st = read_status_api(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_gating(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_conv(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_decode(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_prefill_simt(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_prefill_tc(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_prefill_split(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_decode_step(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_norm(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_mixed(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_prefill_scan(out, clear, s)) != GDN_OK) return st;
    if ((st = read_status_mtp_step(out, clear, s)) != GDN_OK) return st;
    return GDN_OK;
}

gdn_status gdn_state_snapshot(void *pool, int64_t n_slots, int64_t slot_bytes,
                              const int32_t *src, const int32_t *dst, int32_t n,
                              void *stream) {
    GDN_REQUIRE(n >= 0 && n_slots >= 0 && slot_bytes > 0, GDN_ERR_INVALID_ARG);
    if (n == 0) return GDN_OK;
    GDN_REQUIRE(pool && src && dst, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(slot_bytes % 16 == 0 && ((uintptr_t)pool % 16) == 0, GDN_ERR_INVALID_ARG);
    GDN_REQUIRE(n <= 65535, GDN_ERR_UNSUPPORTED);
    const int64_t vecs = slot_bytes / 16;
    const int threads = 256;
    int64_t bx = (vecs + threads * 4 - 1) / (threads * 4);
    if (bx > 1024) bx = 1024;
    if (bx < 1) bx = 1;
    dim3 grid((unsigned)bx, (unsigned)n);
    // programmatic launch: the grid is set up while the kernel before it ends
    const cudaError_t e = launch_after(snapshot_kernel, grid, dim3(threads), 0,
                                       (cudaStream_t)stream, (uint4 *)pool, n_slots, vecs, src, dst);
    if (e != cudaSuccess) {
        set_last_cuda_error(e);
        return GDN_ERR_LAUNCH;
    }
    return GDN_OK;
}

}  // extern "C"

// static_ws.cu -- pa_decode_no_alloc: paged decode whose scratch space is a
// fixed array inside the library instead of memory the caller allocates.
//
// Some callers cannot obtain device memory at the point where they decode: a
// plug-in that runs inside a host framework owning every allocation, a code
// path that must not allocate once serving has started, or an engine that
// carves all of HBM up front and has no spare buffer to hand the library.
// For them the workspace lives in `g_decode_scratch`, a file-scope device
// array that is part of the loaded module, so every GPU that loads libpa.so
// holds it for the life of the process.
#include <mutex>

#include "pa_internal.h"

namespace pa {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_STATIC_WORKSPACE_BYTES];

// In host code `g_decode_scratch` names a host-side stand-in, not device
// memory; the device address comes from cudaGetSymbolAddress, once per device.
constexpr int kMaxDevices = 64;
static std::mutex g_scratch_mu;
static void* g_scratch_ptr[kMaxDevices];

static pa_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static decode workspace)");
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_decode_no_alloc(void* out, pa_dtype out_dtype, const void* q, const void* pool,
                                        const int32_t* block_tables, const int32_t* ctx_lens, int N, int H_q,
                                        int H_kv, int D, int B, int MB, int NB, int max_ctx, float scale,
                                        int partition_tokens, pa_dtype kv_dtype, int* dev_err,
                                        void* const* attend_events, void* stream) {
    const size_t need = pa_decode_workspace_bytes(N, H_q, H_kv, D, max_ctx, partition_tokens);
    if (need == 0) return fail(PA_ERR_INVALID, "invalid sizes or partition_tokens for the decode workspace");
    if (need > (size_t)PA_STATIC_WORKSPACE_BYTES)
        return fail(PA_ERR_UNSUPPORTED,
                    "this batch needs %zu bytes of decode workspace but the built-in workspace holds %zu; "
                    "use pa_decode with a caller-provided workspace (or fewer sequences / a shorter max_ctx)",
                    need, (size_t)PA_STATIC_WORKSPACE_BYTES);
    void* ws = nullptr;
    pa_status st = scratch_address(&ws);
    if (st != PA_OK) return st;
    return pa_decode(out, out_dtype, q, pool, block_tables, ctx_lens, N, H_q, H_kv, D, B, MB, NB, max_ctx, scale,
                     partition_tokens, ws, (size_t)PA_STATIC_WORKSPACE_BYTES, kv_dtype, dev_err, attend_events,
                     stream);
}

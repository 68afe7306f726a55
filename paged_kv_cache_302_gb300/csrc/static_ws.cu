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
#include <cuda.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_STATIC_WORKSPACE_BYTES];

// In host code `g_decode_scratch` names a host-side stand-in, not device
// memory; the device address comes from cudaGetSymbolAddress, called with the
// device current.  The address belongs to the module as loaded into one CUDA
// context, so it is cached per device together with that context's unique ID
// (cuCtxGetId): after cudaDeviceReset, or any other teardown of the context,
// the next call finds a new ID and looks the address up again instead of
// handing the kernels a stale one.
constexpr int kMaxDevices = 64;
static std::mutex g_scratch_mu;
struct ScratchEntry {
    unsigned long long ctx_id;
    void* ptr;
};
static ScratchEntry g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

static void* driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return f;
}

// Unique ID of the context current on this thread (0 when there is none yet).
static pa_status current_ctx_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        get_current = reinterpret_cast<CtxGetCurrentFn>(driver_fn("cuCtxGetCurrent"));
        get_id = reinterpret_cast<CtxGetIdFn>(driver_fn("cuCtxGetId"));
    });
    if (!get_current || !get_id) return fail(PA_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId are not available");
    CUcontext ctx = nullptr;
    CUresult r = get_current(&ctx);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuCtxGetCurrent failed (CUresult %d)", (int)r);
    *id = 0;
    if (ctx) {
        r = get_id(ctx, id);
        if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuCtxGetId failed (CUresult %d)", (int)r);
    }
    return PA_OK;
}

static pa_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    unsigned long long id = 0;
    pa_status st = current_ctx_id(&id);
    if (st != PA_OK) return st;
    ScratchEntry& ent = g_scratch[dev];
    if (id == 0 || ent.ptr == nullptr || ent.ctx_id != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);  // makes the device's primary context current if needed
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static decode workspace)");
        if (id == 0) {
            st = current_ctx_id(&id);
            if (st != PA_OK) return st;
        }
        ent.ctx_id = id;
        ent.ptr = p;
    }
    *out = ent.ptr;
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

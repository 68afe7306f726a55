// vkv.cpp -- virtually contiguous KV buffers backed on demand by physical pages
// (the vAttention explainer, arXiv 2405.04437: 技術的詳細 / CUDA Virtual Memory
// Management APIの活用, 仮想メモリの事前予約, リクエスト単位のKVキャッシュインデキシング;
// 実装のポイント for the init / alloc_reqid / step / free_reqid interface).
//
// Every K (and V) buffer of every layer is one reserved virtual range of
// max_batch request regions; request r's cache starts at r * S.  Physical
// pages (the driver's allocation granularity, 2 MB here) are created and mapped
// only when a request's context grows into them; a freed request slot keeps its
// pages (deferred reclamation) and the next owner of the slot reuses them.
#include <cuda.h>

#include <algorithm>
#include <mutex>
#include <new>
#include <numeric>
#include <vector>

#include "pa_internal.h"

namespace pa {

namespace {

struct DriverVmm {
    CUresult (*granularity)(size_t*, const CUmemAllocationProp*, CUmemAllocationGranularity_flags) = nullptr;
    CUresult (*reserve)(CUdeviceptr*, size_t, size_t, CUdeviceptr, unsigned long long) = nullptr;
    CUresult (*addr_free)(CUdeviceptr, size_t) = nullptr;
    CUresult (*create)(CUmemGenericAllocationHandle*, size_t, const CUmemAllocationProp*, unsigned long long) =
        nullptr;
    CUresult (*release)(CUmemGenericAllocationHandle) = nullptr;
    CUresult (*map)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle, unsigned long long) = nullptr;
    CUresult (*unmap)(CUdeviceptr, size_t) = nullptr;
    CUresult (*set_access)(CUdeviceptr, size_t, const CUmemAccessDesc*, size_t) = nullptr;
    bool ok = false;
};

const DriverVmm& vmm() {
    static DriverVmm d;
    static std::once_flag once;
    std::call_once(once, [] {
        auto get = [](const char* name, void** fn) {
            cudaDriverEntryPointQueryResult q;
            return cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                   q == cudaDriverEntryPointSuccess && *fn;
        };
        d.ok = get("cuMemGetAllocationGranularity", reinterpret_cast<void**>(&d.granularity)) &&
               get("cuMemAddressReserve", reinterpret_cast<void**>(&d.reserve)) &&
               get("cuMemAddressFree", reinterpret_cast<void**>(&d.addr_free)) &&
               get("cuMemCreate", reinterpret_cast<void**>(&d.create)) &&
               get("cuMemRelease", reinterpret_cast<void**>(&d.release)) &&
               get("cuMemMap", reinterpret_cast<void**>(&d.map)) &&
               get("cuMemUnmap", reinterpret_cast<void**>(&d.unmap)) &&
               get("cuMemSetAccess", reinterpret_cast<void**>(&d.set_access));
    });
    return d;
}

// Tokens a decode stage reads at once (the attention kernel's TMA box): a
// request's mapping always covers its context rounded up to this.
constexpr int kReadGranule = kStageTok;

}  // namespace

struct Vkv {
    int layers = 0, max_batch = 0, max_ctx = 0, H_kv = 0, D = 0, device = 0;
    size_t row_bytes = 0;     // one token of one head group: H_kv * D * elem
    size_t page = 0;          // physical page size (allocation granularity)
    size_t per_req = 0;       // bytes of one request region, a multiple of page and of row_bytes
    int64_t S_tokens = 0;     // per_req / row_bytes: the request stride in tokens
    size_t buf_bytes = 0;     // max_batch * per_req
    std::vector<CUdeviceptr> base;                           // [2 * layers]: K then V of each layer
    std::vector<int> pages;                                  // [max_batch]: pages mapped per region
    std::vector<std::vector<CUmemGenericAllocationHandle>> handles;  // [2 * layers * max_batch]
    std::vector<char> used;                                  // [max_batch]
    CUmemAllocationProp prop{};
    CUmemAccessDesc access{};
};

static Vkv* as_vkv(void* h) { return static_cast<Vkv*>(h); }

static pa_status drv_fail(CUresult r, const char* what) {
    return fail(r == CUDA_ERROR_OUT_OF_MEMORY ? PA_ERR_OOM : PA_ERR_CUDA, "%s failed (CUresult %d)", what, (int)r);
}

// Unmaps and releases pages [from, to) of request region r in every buffer.
static void unmap_pages(Vkv& V, int r, int from, int to) {
    const DriverVmm& d = vmm();
    for (size_t b = 0; b < V.base.size(); ++b) {
        auto& hs = V.handles[b * V.max_batch + r];
        for (int pg = std::min<int>(to, (int)hs.size()) - 1; pg >= from; --pg) {
            const CUdeviceptr va = V.base[b] + (CUdeviceptr)r * V.per_req + (CUdeviceptr)pg * V.page;
            d.unmap(va, V.page);
            d.release(hs[pg]);
            hs.pop_back();
        }
    }
}

// Maps pages so region r covers `tokens` tokens in every buffer; all or nothing.
static pa_status map_to(Vkv& V, int r, int64_t tokens) {
    const DriverVmm& d = vmm();
    const int64_t need = ((int64_t)tokens * (int64_t)V.row_bytes + (int64_t)V.page - 1) / (int64_t)V.page;
    const int have = V.pages[r];
    for (int pg = have; pg < need; ++pg) {
        for (size_t b = 0; b < V.base.size(); ++b) {
            CUmemGenericAllocationHandle h;
            CUresult res = d.create(&h, V.page, &V.prop, 0);
            pa_status st = PA_OK;
            if (res != CUDA_SUCCESS) {
                st = drv_fail(res, "cuMemCreate");
            } else {
                const CUdeviceptr va = V.base[b] + (CUdeviceptr)r * V.per_req + (CUdeviceptr)pg * V.page;
                res = d.map(va, V.page, 0, h, 0);
                if (res == CUDA_SUCCESS) res = d.set_access(va, V.page, &V.access, 1);
                if (res != CUDA_SUCCESS) {
                    d.unmap(va, V.page);
                    d.release(h);
                    st = drv_fail(res, "cuMemMap / cuMemSetAccess");
                } else {
                    V.handles[b * V.max_batch + r].push_back(h);
                }
            }
            if (st != PA_OK) {
                // undo this call: buffers before b got page pg, all buffers got pages [have, pg)
                for (size_t bb = 0; bb < b; ++bb) {
                    auto& hs = V.handles[bb * V.max_batch + r];
                    const CUdeviceptr va = V.base[bb] + (CUdeviceptr)r * V.per_req + (CUdeviceptr)pg * V.page;
                    d.unmap(va, V.page);
                    d.release(hs.back());
                    hs.pop_back();
                }
                unmap_pages(V, r, have, pg);
                V.pages[r] = have;
                return st;
            }
        }
        V.pages[r] = pg + 1;
    }
    return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" {

pa_status pa_vkv_create(int num_layers, int max_batch, int max_ctx, int H_kv, int D, pa_dtype dtype, void** out) {
    if (!out) return fail(PA_ERR_INVALID, "out is null");
    *out = nullptr;
    if (num_layers <= 0 || max_batch <= 0 || max_ctx <= 0 || H_kv <= 0 || D <= 0)
        return fail(PA_ERR_INVALID, "sizes must be positive");
    if (dtype != PA_F16 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "dtype must be F16 or BF16");
    const DriverVmm& d = vmm();
    if (!d.ok) return fail(PA_ERR_CUDA, "the driver's virtual memory management calls are not available");
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess) return cuda_fail(ce, "cudaGetDevice");
    Vkv* V = new (std::nothrow) Vkv;
    if (!V) return fail(PA_ERR_OOM, "host allocation failed");
    V->layers = num_layers;
    V->max_batch = max_batch;
    V->max_ctx = max_ctx;
    V->H_kv = H_kv;
    V->D = D;
    V->device = dev;
    V->row_bytes = (size_t)H_kv * D * 2;
    V->prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    V->prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    V->prop.location.id = dev;
    V->access.location = V->prop.location;
    V->access.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    CUresult r = d.granularity(&V->page, &V->prop, CU_MEM_ALLOC_GRANULARITY_MINIMUM);
    if (r != CUDA_SUCCESS || V->page == 0) {
        delete V;
        return drv_fail(r, "cuMemGetAllocationGranularity");
    }
    // a request region: whole pages and whole tokens, holding max_ctx tokens rounded up to the read granule
    const size_t unit = std::lcm(V->page, V->row_bytes * kReadGranule);
    const size_t want = (size_t)((max_ctx + kReadGranule - 1) / kReadGranule * kReadGranule) * V->row_bytes;
    V->per_req = (want + unit - 1) / unit * unit;
    V->S_tokens = (int64_t)(V->per_req / V->row_bytes);
    V->buf_bytes = (size_t)max_batch * V->per_req;
    if ((int64_t)max_batch * V->S_tokens >= (1LL << 31)) {
        delete V;
        return fail(PA_ERR_UNSUPPORTED, "max_batch * tokens per region must be < 2^31");
    }
    V->pages.assign(max_batch, 0);
    V->used.assign(max_batch, 0);
    V->handles.resize((size_t)2 * num_layers * max_batch);
    for (int b = 0; b < 2 * num_layers; ++b) {
        CUdeviceptr p = 0;
        r = d.reserve(&p, V->buf_bytes, V->page, 0, 0);
        if (r != CUDA_SUCCESS) {
            for (CUdeviceptr q : V->base) d.addr_free(q, V->buf_bytes);
            delete V;
            return drv_fail(r, "cuMemAddressReserve");
        }
        V->base.push_back(p);
    }
    *out = V;
    return PA_OK;
}

void pa_vkv_destroy(void* h) {
    Vkv* V = as_vkv(h);
    if (!V) return;
    for (int r = 0; r < V->max_batch; ++r) unmap_pages(*V, r, 0, V->pages[r]);
    for (CUdeviceptr p : V->base) vmm().addr_free(p, V->buf_bytes);
    delete V;
}

pa_status pa_vkv_info(void* h, void** k_bufs, void** v_bufs, int64_t* S_tokens, int64_t* page_bytes) {
    Vkv* V = as_vkv(h);
    if (!V) return fail(PA_ERR_INVALID, "null handle");
    for (int l = 0; l < V->layers; ++l) {
        if (k_bufs) k_bufs[l] = reinterpret_cast<void*>(V->base[2 * l]);
        if (v_bufs) v_bufs[l] = reinterpret_cast<void*>(V->base[2 * l + 1]);
    }
    if (S_tokens) *S_tokens = V->S_tokens;
    if (page_bytes) *page_bytes = (int64_t)V->page;
    return PA_OK;
}

pa_status pa_vkv_alloc_reqid(void* h, int* req_id) {
    Vkv* V = as_vkv(h);
    if (!V || !req_id) return fail(PA_ERR_INVALID, "null argument");
    // prefer a free slot whose pages are still mapped (deferred reclamation), then the lowest id
    int best = -1;
    for (int r = 0; r < V->max_batch; ++r)
        if (!V->used[r] && (best < 0 || V->pages[r] > V->pages[best])) best = r;
    if (best < 0) return fail(PA_ERR_OOM, "all %d request slots are in use", V->max_batch);
    V->used[best] = 1;
    *req_id = best;
    return PA_OK;
}

pa_status pa_vkv_step(void* h, const int32_t* req_ids, const int32_t* ctx_lens, int n) {
    Vkv* V = as_vkv(h);
    if (!V) return fail(PA_ERR_INVALID, "null handle");
    if (n < 0 || (n > 0 && (!req_ids || !ctx_lens))) return fail(PA_ERR_INVALID, "bad arguments");
    for (int i = 0; i < n; ++i) {
        if (req_ids[i] < 0 || req_ids[i] >= V->max_batch || !V->used[req_ids[i]])
            return fail(PA_ERR_INVALID, "request %d is not allocated", req_ids[i]);
        if (ctx_lens[i] < 0 || ctx_lens[i] > V->max_ctx)
            return fail(PA_ERR_INVALID, "context %d outside [0, %d]", ctx_lens[i], V->max_ctx);
    }
    int dev_now = 0;
    cudaGetDevice(&dev_now);
    if (dev_now != V->device) return fail(PA_ERR_INVALID, "call with device %d current", V->device);
    for (int i = 0; i < n; ++i) {
        const int64_t cover = ((int64_t)ctx_lens[i] + kReadGranule - 1) / kReadGranule * kReadGranule;
        pa_status st = map_to(*V, req_ids[i], cover);
        if (st != PA_OK) return st;  // earlier requests keep their (valid) new pages
    }
    return PA_OK;
}

pa_status pa_vkv_free_reqid(void* h, int req_id) {
    Vkv* V = as_vkv(h);
    if (!V) return fail(PA_ERR_INVALID, "null handle");
    if (req_id < 0 || req_id >= V->max_batch || !V->used[req_id])
        return fail(PA_ERR_INVALID, "request %d is not allocated", req_id);
    V->used[req_id] = 0;  // pages stay mapped for the slot's next owner
    return PA_OK;
}

pa_status pa_vkv_reclaim(void* h) {
    Vkv* V = as_vkv(h);
    if (!V) return fail(PA_ERR_INVALID, "null handle");
    for (int r = 0; r < V->max_batch; ++r)
        if (!V->used[r]) {
            unmap_pages(*V, r, 0, V->pages[r]);
            V->pages[r] = 0;
        }
    return PA_OK;
}

pa_status pa_vkv_mapped_pages(void* h, int req_id, int* pages) {
    Vkv* V = as_vkv(h);
    if (!V || !pages) return fail(PA_ERR_INVALID, "null argument");
    if (req_id < 0 || req_id >= V->max_batch) return fail(PA_ERR_INVALID, "request %d out of range", req_id);
    *pages = V->pages[req_id];
    return PA_OK;
}

}  // extern "C"

// capi.cpp -- argument validation and dispatch for the device entry points of pa.h.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <nvtx3/nvToolsExt.h>

#include "pa_internal.h"

namespace pa {

static thread_local char g_msg[512] = "";
static std::atomic<uint64_t> g_launches{0};

pa_status fail(pa_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return st;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static std::atomic<uint64_t> g_wait_ns{0};  // 0: the built-in limit

uint64_t wait_limit_ns() {
    const uint64_t ns = g_wait_ns.load(std::memory_order_relaxed);
    return ns ? ns : 1000000000ull;
}

// NVTX ranges around every device call, for profiler timelines; off unless PA_NVTX is set to a non-zero value
// (read once), so a call costs one predictable branch when they are off.
static bool nvtx_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("PA_NVTX");
        return v && *v && *v != '0';
    }();
    return on;
}

struct NvtxRange {
    bool on;
    explicit NvtxRange(const char* name) : on(nvtx_enabled()) {
        if (on) nvtxRangePushA(name);
    }
    ~NvtxRange() {
        if (on) nvtxRangePop();
    }
};

bool pdl_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("PA_NO_PDL");
        return !(v && *v && *v != '0');
    }();
    return on;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool kv_dtype_ok(int dt) { return dt == PA_F16 || dt == PA_BF16; }

static pa_status check_decode_common(pa_dtype out_dtype, pa_dtype kv_dtype, const void* out, const void* q,
                                     const int32_t* ctx_lens, int N, int H_q, int H_kv, int D, int max_ctx,
                                     int partition_tokens, const void* ws, size_t ws_bytes) {
    if (!kv_dtype_ok(kv_dtype)) return fail(PA_ERR_UNSUPPORTED, "kv_dtype must be F16 or BF16");
    if (out_dtype != PA_F32 && out_dtype != kv_dtype)
        return fail(PA_ERR_UNSUPPORTED, "out_dtype must be F32 or the kv dtype");
    if (N <= 0 || H_q <= 0 || H_kv <= 0 || max_ctx <= 0) return fail(PA_ERR_INVALID, "sizes must be positive");
    if (H_q % H_kv) return fail(PA_ERR_INVALID, "H_q (%d) must be a multiple of H_kv (%d)", H_q, H_kv);
    if (H_q / H_kv > kMaxGroup) return fail(PA_ERR_UNSUPPORTED, "H_q / H_kv must be <= %d", kMaxGroup);
    if (D != 64 && D != 128) return fail(PA_ERR_UNSUPPORTED, "D must be 64 or 128 (got %d)", D);
    if (!out || !q || !ctx_lens || !ws) return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(out) || !aligned16(q) || !aligned16(ws))
        return fail(PA_ERR_INVALID, "out, q and workspace must be 16-byte aligned");
    WorkspaceLayout L;
    if (!workspace_layout(N, H_q, H_kv, D, max_ctx, partition_tokens, &L))
        return fail(PA_ERR_INVALID, "partition_tokens must be 0, -1 or a positive multiple of %d", kStageTok);
    if (ws_bytes < L.total) return fail(PA_ERR_INVALID, "workspace too small: %zu < %zu bytes", ws_bytes, L.total);
    if ((long)N * L.P * H_kv >= (1L << 30)) return fail(PA_ERR_UNSUPPORTED, "too many work records");
    return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_last_error(void) { return g_msg; }

const char* pa_version(void) { return "pa 0.1.0 (sm_103a)"; }

uint64_t pa_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

void pa_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns, std::memory_order_relaxed); }

pa_status pa_reshape_and_cache(const void* k, const void* v, void* pool, const int64_t* slot_mapping, int T, int NB,
                               int B, int H_kv, int D, pa_dtype dtype, int* dev_err, void* stream) {
    const NvtxRange nvtx_range("pa_reshape_and_cache");
    g_msg[0] = 0;
    if (!kv_dtype_ok(dtype)) return fail(PA_ERR_UNSUPPORTED, "dtype must be F16 or BF16");
    if (T < 0 || NB <= 0 || B <= 0 || H_kv <= 0 || D <= 0) return fail(PA_ERR_INVALID, "bad sizes");
    if ((H_kv * D) % 8) return fail(PA_ERR_UNSUPPORTED, "H_kv * D must be a multiple of 8");
    if ((long long)NB * B >= (1LL << 62)) return fail(PA_ERR_INVALID, "pool too large");
    if (T == 0) return PA_OK;
    if (!k || !v || !pool || !slot_mapping) return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(k) || !aligned16(v) || !aligned16(pool))
        return fail(PA_ERR_INVALID, "k, v and pool must be 16-byte aligned");
    return launch_reshape_and_cache(k, v, pool, slot_mapping, T, NB, B, H_kv, D, dev_err,
                                    static_cast<cudaStream_t>(stream));
}

pa_status pa_copy_blocks(void* pool, const int64_t* pairs, int n, int NB, int B, int H_kv, int D, pa_dtype dtype,
                         int* dev_err, void* stream) {
    const NvtxRange nvtx_range("pa_copy_blocks");
    g_msg[0] = 0;
    if (!kv_dtype_ok(dtype)) return fail(PA_ERR_UNSUPPORTED, "dtype must be F16 or BF16");
    if (n < 0 || NB <= 0 || B <= 0 || H_kv <= 0 || D <= 0) return fail(PA_ERR_INVALID, "bad sizes");
    if (((long long)B * 2 * H_kv * D * 2) % 16) return fail(PA_ERR_UNSUPPORTED, "block bytes must be a multiple of 16");
    if (n > (1 << 30)) return fail(PA_ERR_INVALID, "too many pairs");
    if (n == 0) return PA_OK;
    if (!pool || !pairs) return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(pool)) return fail(PA_ERR_INVALID, "pool must be 16-byte aligned");
    return launch_copy_blocks(pool, pairs, n, NB, B, H_kv, D, dev_err, static_cast<cudaStream_t>(stream));
}

// A pointer the GPU may dereference: device memory, managed memory, or page-locked host memory.
static pa_status check_device_accessible(const void* p, const char* what) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
    if (attr.type == cudaMemoryTypeUnregistered)
        return fail(PA_ERR_INVALID, "%s is pageable host memory; pin it (cudaHostAlloc / cudaHostRegister)", what);
    if (attr.type == cudaMemoryTypeHost && !attr.devicePointer)
        return fail(PA_ERR_INVALID, "%s is page-locked but not mapped into the device address space", what);
    return PA_OK;
}

pa_status pa_swap_blocks(void* dst_pool, int NB_dst, const void* src_pool, int NB_src, const int64_t* pairs, int n,
                         int B, int H_kv, int D, pa_dtype dtype, int* dev_err, void* stream) {
    const NvtxRange nvtx_range("pa_swap_blocks");
    g_msg[0] = 0;
    if (!kv_dtype_ok(dtype)) return fail(PA_ERR_UNSUPPORTED, "dtype must be F16 or BF16");
    if (n < 0 || NB_dst <= 0 || NB_src <= 0 || B <= 0 || H_kv <= 0 || D <= 0) return fail(PA_ERR_INVALID, "bad sizes");
    const long long blk_bytes = (long long)B * 2 * H_kv * D * 2;
    if (blk_bytes % 16) return fail(PA_ERR_UNSUPPORTED, "block bytes must be a multiple of 16");
    if (n > (1 << 30)) return fail(PA_ERR_INVALID, "too many pairs");
    if (n == 0) return PA_OK;
    if (!dst_pool || !src_pool || !pairs) return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(dst_pool) || !aligned16(src_pool)) return fail(PA_ERR_INVALID, "pools must be 16-byte aligned");
    pa_status st = check_device_accessible(dst_pool, "dst_pool");
    if (st == PA_OK) st = check_device_accessible(src_pool, "src_pool");
    if (st == PA_OK) st = check_device_accessible(pairs, "pairs");
    if (st != PA_OK) return st;
    return launch_swap_blocks(dst_pool, NB_dst, src_pool, NB_src, pairs, n, blk_bytes, dev_err,
                              static_cast<cudaStream_t>(stream));
}

pa_status pa_write_contiguous(const void* k, const void* v, void* k_buf, void* v_buf, const int32_t* req_ids,
                              const int32_t* positions, int T, int N_max, int S_max, int H_kv, int D, pa_dtype dtype,
                              int* dev_err, void* stream) {
    const NvtxRange nvtx_range("pa_write_contiguous");
    g_msg[0] = 0;
    if (!kv_dtype_ok(dtype)) return fail(PA_ERR_UNSUPPORTED, "dtype must be F16 or BF16");
    if (T < 0 || N_max <= 0 || S_max <= 0 || H_kv <= 0 || D <= 0) return fail(PA_ERR_INVALID, "bad sizes");
    if ((H_kv * D) % 8) return fail(PA_ERR_UNSUPPORTED, "H_kv * D must be a multiple of 8");
    if (T == 0) return PA_OK;
    if (!k || !v || !k_buf || !v_buf || !req_ids || !positions) return fail(PA_ERR_INVALID, "null pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_buf) || !aligned16(v_buf))
        return fail(PA_ERR_INVALID, "k, v and the buffers must be 16-byte aligned");
    return launch_write_contiguous(k, v, k_buf, v_buf, req_ids, positions, T, N_max, S_max, H_kv, D, dev_err,
                                   static_cast<cudaStream_t>(stream));
}

pa_status pa_update_block_tables(int32_t* tables, int N, int MB, const int32_t* updates, int n, int* dev_err,
                                 void* stream) {
    const NvtxRange nvtx_range("pa_update_block_tables");
    g_msg[0] = 0;
    if (N <= 0 || MB <= 0 || n < 0) return fail(PA_ERR_INVALID, "bad sizes");
    if (n == 0) return PA_OK;
    if (!tables || !updates) return fail(PA_ERR_INVALID, "null pointer argument");
    if ((reinterpret_cast<uintptr_t>(updates) & 3u) || (reinterpret_cast<uintptr_t>(tables) & 3u))
        return fail(PA_ERR_INVALID, "tables and updates must be 4-byte aligned");
    return launch_update_tables(tables, N, MB, updates, n, dev_err, static_cast<cudaStream_t>(stream));
}

size_t pa_decode_workspace_bytes(int N, int H_q, int H_kv, int D, int max_ctx, int partition_tokens) {
    WorkspaceLayout L;
    if (!workspace_layout(N, H_q, H_kv, D, max_ctx, partition_tokens, &L)) return 0;
    return L.total;
}

pa_status pa_decode(void* out, pa_dtype out_dtype, const void* q, const void* pool, const int32_t* block_tables,
                    const int32_t* ctx_lens, int N, int H_q, int H_kv, int D, int B, int MB, int NB, int max_ctx,
                    float scale, int partition_tokens, void* workspace, size_t ws_bytes, pa_dtype kv_dtype,
                    int* dev_err, void* const* attend_events, void* stream) {
    const NvtxRange nvtx_range("pa_decode");
    g_msg[0] = 0;
    pa_status st = check_decode_common(out_dtype, kv_dtype, out, q, ctx_lens, N, H_q, H_kv, D, max_ctx,
                                       partition_tokens, workspace, ws_bytes);
    if (st != PA_OK) return st;
    if (B != 4 && B != 8 && B != 16 && B != 32) return fail(PA_ERR_UNSUPPORTED, "B must be 4, 8, 16 or 32");
    if (NB <= 0 || MB <= 0) return fail(PA_ERR_INVALID, "NB and MB must be positive");
    if ((long long)NB * B >= (1LL << 31)) return fail(PA_ERR_UNSUPPORTED, "NB * B must be < 2^31");
    if (!pool || !block_tables) return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(pool)) return fail(PA_ERR_INVALID, "pool must be 16-byte aligned");
    DecodeArgs a;
    std::memset(&a, 0, sizeof a);
    a.out = out;
    a.out_dtype = out_dtype;
    a.q = q;
    a.kv_dtype = kv_dtype;
    a.pool = pool;
    a.tables = block_tables;
    a.B = B;
    a.MB = MB;
    a.NB = NB;
    a.paged = true;
    a.ctx_lens = ctx_lens;
    a.N = N;
    a.H_q = H_q;
    a.H_kv = H_kv;
    a.D = D;
    a.max_ctx = max_ctx;
    a.scale = scale;
    a.partition_tokens = partition_tokens;
    a.workspace = workspace;
    a.ws_bytes = ws_bytes;
    a.dev_err = dev_err;
    a.attend_events = attend_events;
    a.stream = static_cast<cudaStream_t>(stream);
    return launch_decode(a);
}

pa_status pa_decode_contiguous(void* out, pa_dtype out_dtype, const void* q, const void* k_buf, const void* v_buf,
                               const int32_t* req_ids, const int32_t* ctx_lens, int N, int H_q, int H_kv, int D,
                               int N_max, int S_max, int max_ctx, float scale, int partition_tokens, void* workspace,
                               size_t ws_bytes, pa_dtype kv_dtype, int* dev_err, void* const* attend_events,
                               void* stream) {
    const NvtxRange nvtx_range("pa_decode_contiguous");
    g_msg[0] = 0;
    pa_status st = check_decode_common(out_dtype, kv_dtype, out, q, ctx_lens, N, H_q, H_kv, D, max_ctx,
                                       partition_tokens, workspace, ws_bytes);
    if (st != PA_OK) return st;
    if (N_max <= 0 || S_max <= 0) return fail(PA_ERR_INVALID, "N_max and S_max must be positive");
    if ((long long)N_max * S_max >= (1LL << 31)) return fail(PA_ERR_UNSUPPORTED, "N_max * S_max must be < 2^31");
    if (!k_buf || !v_buf || !req_ids) return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(k_buf) || !aligned16(v_buf)) return fail(PA_ERR_INVALID, "k_buf and v_buf must be 16-byte aligned");
    DecodeArgs a;
    std::memset(&a, 0, sizeof a);
    a.out = out;
    a.out_dtype = out_dtype;
    a.q = q;
    a.kv_dtype = kv_dtype;
    a.k_buf = k_buf;
    a.v_buf = v_buf;
    a.req_ids = req_ids;
    a.N_max = N_max;
    a.S_max = S_max;
    a.paged = false;
    a.ctx_lens = ctx_lens;
    a.N = N;
    a.H_q = H_q;
    a.H_kv = H_kv;
    a.D = D;
    a.max_ctx = max_ctx;
    a.scale = scale;
    a.partition_tokens = partition_tokens;
    a.workspace = workspace;
    a.ws_bytes = ws_bytes;
    a.dev_err = dev_err;
    a.attend_events = attend_events;
    a.stream = static_cast<cudaStream_t>(stream);
    return launch_decode(a);
}

size_t pa_prefill_workspace_bytes(int N, int H_kv, int D, int B, int MB) {
    PrefillWorkspace L;
    return prefill_workspace_layout(N, H_kv, D, B, MB, &L) ? L.total : 0;
}

pa_status pa_prefill(void* out, pa_dtype out_dtype, const void* q, const void* pool, const int32_t* block_tables,
                     const int32_t* ctx_lens, const int32_t* q_start, int N, int T, int H_q, int H_kv, int D, int B,
                     int MB, int NB, int max_q_len, float scale, pa_dtype kv_dtype, void* workspace, size_t ws_bytes,
                     int* dev_err, void* stream) {
    const NvtxRange nvtx_range("pa_prefill");
    g_msg[0] = 0;
    if (!kv_dtype_ok(kv_dtype)) return fail(PA_ERR_UNSUPPORTED, "kv_dtype must be F16 or BF16");
    if (out_dtype != PA_F32 && out_dtype != kv_dtype)
        return fail(PA_ERR_UNSUPPORTED, "out_dtype must be F32 or the kv dtype");
    if (N <= 0 || N > 65535 || T < 0 || H_q <= 0 || H_kv <= 0 || H_kv > 65535 || MB <= 0 || NB <= 0 ||
        max_q_len < 0)
        return fail(PA_ERR_INVALID, "bad sizes");
    if (H_q % H_kv) return fail(PA_ERR_INVALID, "H_q must be a multiple of H_kv");
    if (H_q / H_kv > 128) return fail(PA_ERR_UNSUPPORTED, "H_q / H_kv must be <= 128");
    if (D != 64 && D != 128) return fail(PA_ERR_UNSUPPORTED, "D must be 64 or 128");
    if (B != 8 && B != 16 && B != 32) return fail(PA_ERR_UNSUPPORTED, "prefill supports B in {8, 16, 32}");
    if (!(scale > 0.f)) return fail(PA_ERR_INVALID, "scale must be positive");
    if ((long long)NB * B >= (1LL << 31)) return fail(PA_ERR_UNSUPPORTED, "NB * B must be < 2^31");
    if (T == 0 || max_q_len == 0) return PA_OK;
    if (!out || !q || !pool || !block_tables || !ctx_lens || !q_start) return fail(PA_ERR_INVALID, "null pointer");
    if (!aligned16(out) || !aligned16(q) || !aligned16(pool) || !aligned16(workspace))
        return fail(PA_ERR_INVALID, "16-byte alignment");
    if (out_dtype == PA_F32 && (reinterpret_cast<uintptr_t>(out) & 31u))
        return fail(PA_ERR_INVALID, "an fp32 out must be 32-byte aligned");
    PrefillArgs a;
    a.out = out;
    a.out_dtype = out_dtype;
    a.q = q;
    a.pool = pool;
    a.tables = block_tables;
    a.ctx_lens = ctx_lens;
    a.q_start = q_start;
    a.N = N;
    a.T = T;
    a.H_q = H_q;
    a.H_kv = H_kv;
    a.D = D;
    a.B = B;
    a.MB = MB;
    a.NB = NB;
    a.max_q_len = max_q_len;
    a.scale = scale;
    a.kv_dtype = kv_dtype;
    a.workspace = workspace;
    a.ws_bytes = workspace ? ws_bytes : 0;
    a.dev_err = dev_err;
    a.stream = static_cast<cudaStream_t>(stream);
    return launch_prefill(a);
}

pa_status pa_partition_reduce(void* out, pa_dtype out_dtype, const float* part_m2, const float* part_l,
                              const float* part_acc, const int32_t* nparts, int R, int P, int D, int* dev_err,
                              void* stream) {
    const NvtxRange nvtx_range("pa_partition_reduce");
    g_msg[0] = 0;
    if (out_dtype != PA_F32 && out_dtype != PA_F16 && out_dtype != PA_BF16)
        return fail(PA_ERR_UNSUPPORTED, "bad out_dtype");
    if (D != 64 && D != 128) return fail(PA_ERR_UNSUPPORTED, "D must be 64 or 128");
    if (R < 0 || P <= 0) return fail(PA_ERR_INVALID, "bad sizes");
    if (R == 0) return PA_OK;
    if (!out || !part_m2 || !part_l || !part_acc || !nparts) return fail(PA_ERR_INVALID, "null pointer argument");
    if (!aligned16(part_acc)) return fail(PA_ERR_INVALID, "part_acc must be 16-byte aligned");
    return launch_partition_reduce(out, out_dtype, part_m2, part_l, part_acc, nparts, 1, R, P, D, false, dev_err,
                                   static_cast<cudaStream_t>(stream));
}

}  // extern "C"

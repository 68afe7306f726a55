// cache_ops.cu -- cache write through slot_mapping and copy-on-write block copy.
//
// Both are bit copies of 16-byte vectors; neither converts or interprets the
// elements.  Sources: PagedAttention explainer (0h-n0.github.io, arXiv
// 2309.06180), 技術的詳細 / PagedAttentionアルゴリズム (tokens stored in fixed-size
// blocks reached through a block table) and Copy-on-Write KVキャッシュ共有 (copy a
// shared block before writing into it).
#include "pa_device.cuh"

namespace pa {

// Grid of a per-token copy: one CTA per token up to 16 resident CTAs per SM of the current device.
static int token_grid(int T) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                  cudaSuccess || sms < 1)
        sms = 1;
    const long cap = 16L * sms;
    return T < cap ? T : (int)cap;
}

// One CTA per token (grid-stride).  Token i's K row and V row (H_kv*D elements
// each, contiguous in both source and pool) are copied to slot slots[i].
__global__ void __launch_bounds__(128) reshape_and_cache_kernel(const uint4* __restrict__ k,
                                                                const uint4* __restrict__ v, uint4* __restrict__ pool,
                                                                const int64_t* __restrict__ slots, int T,
                                                                int64_t nslots, int row_vec, int B, int* err) {
    griddep_wait();
    griddep_launch_dependents();
    for (int i = blockIdx.x; i < T; i += gridDim.x) {
        const int64_t slot = slots[i];
        if (slot < 0) continue;
        if (slot >= nslots) {
            if (threadIdx.x == 0) flag_error(err, PA_DEV_ERR_SLOT);
            continue;
        }
        const int64_t blk = slot / B, off = slot - blk * B;
        uint4* dk = pool + (blk * B + off) * 2 * (int64_t)row_vec;
        uint4* dv = dk + row_vec;
        const uint4* sk = k + (int64_t)i * row_vec;
        const uint4* sv = v + (int64_t)i * row_vec;
        for (int e = threadIdx.x; e < row_vec; e += blockDim.x) {
            const uint4 a = sk[e];
            const uint4 b = sv[e];
            dk[e] = a;
            dv[e] = b;
        }
    }
}

pa_status launch_reshape_and_cache(const void* k, const void* v, void* pool, const int64_t* slot_mapping, int T,
                                   int NB, int B, int H_kv, int D, int* dev_err, cudaStream_t stream) {
    if (T == 0) return PA_OK;
    const int row_vec = H_kv * D * 2 / 16;
    const int grid = token_grid(T);
    cudaError_t e = launch_kernel(reshape_and_cache_kernel, dim3(grid), dim3(128), 0, stream,
                                  static_cast<const uint4*>(k), static_cast<const uint4*>(v),
                                  static_cast<uint4*>(pool), slot_mapping, T, (int64_t)NB * B, row_vec, B, dev_err);
    count_launch();
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "reshape_and_cache launch");
}

// grid.x = pair index (plus the check CTAs below), grid.y = chunk of the block; each thread moves kUnroll vectors
// per chunk with all loads issued before the stores.
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

// Chained pairs (a destination that is also a source, or a destination named twice) make the result of a copy
// call depend on the order of the copies; they are flagged, in one pass over the pairs, by kCheckIds-wide ranges
// of block ids: check CTA r (grid.x = n + r, grid.y = 0) marks the destinations that fall in its range in a
// shared-memory bitmap (a bit found already set is a repeated destination), then looks up the sources in its
// range.  One check CTA covers 131072 block ids; the check runs beside the copies, in the same launch.
constexpr int kCheckWords = 4096;  // 16 KB of bitmap
constexpr int64_t kCheckIds = (int64_t)kCheckWords * 32;

__device__ __forceinline__ void check_pairs(const int64_t* __restrict__ pairs, int n, int64_t lo, uint32_t* bits,
                                            int* err) {
    for (int i = threadIdx.x; i < kCheckWords; i += blockDim.x) bits[i] = 0;
    __syncthreads();
    bool bad = false;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int64_t d = pairs[2 * i + 1] - lo;
        if (d >= 0 && d < kCheckIds) {
            const uint32_t m = 1u << (d & 31);
            if (atomicOr(&bits[d >> 5], m) & m) bad = true;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int64_t s = pairs[2 * i] - lo;
        if (s >= 0 && s < kCheckIds && (bits[s >> 5] >> (s & 31)) & 1u) bad = true;
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_error(err, PA_DEV_ERR_BLOCK);
}

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(uint4* __restrict__ pool,
                                                                   const int64_t* __restrict__ pairs, int n, int NB,
                                                                   int64_t blk_vec, int* err) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ uint32_t bits[kCheckWords];
    const int i = blockIdx.x;
    if (i >= n) {
        if (blockIdx.y == 0) check_pairs(pairs, n, (int64_t)(i - n) * kCheckIds, bits, err);
        return;
    }
    const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
    if (src < 0 || src >= NB || dst < 0 || dst >= NB) {
        if (threadIdx.x == 0 && blockIdx.y == 0) flag_error(err, PA_DEV_ERR_BLOCK);
        return;
    }
    const uint4* s = pool + src * blk_vec;
    uint4* d = pool + dst * blk_vec;
    const int64_t chunk = (int64_t)kCopyThreads * kCopyUnroll;
    for (int64_t base = (int64_t)blockIdx.y * chunk; base < blk_vec; base += (int64_t)gridDim.y * chunk) {
        uint4 r[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t e = base + u * kCopyThreads + threadIdx.x;
            if (e < blk_vec) r[u] = s[e];
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t e = base + u * kCopyThreads + threadIdx.x;
            if (e < blk_vec) d[e] = r[u];
        }
    }
}

pa_status launch_copy_blocks(void* pool, const int64_t* pairs, int n, int NB, int B, int H_kv, int D, int* dev_err,
                             cudaStream_t stream) {
    if (n == 0) return PA_OK;
    const int64_t blk_vec = (int64_t)B * 2 * H_kv * D * 2 / 16;
    const int64_t chunk = (int64_t)kCopyThreads * kCopyUnroll;
    int64_t gy = (blk_vec + chunk - 1) / chunk;
    if (gy > 65535) gy = 65535;
    const int64_t gx = (int64_t)n + ((int64_t)NB + kCheckIds - 1) / kCheckIds;
    if (gx > 0x7fffffff) return fail(PA_ERR_INVALID, "too many copy pairs: %d", n);
    cudaError_t e = launch_kernel(copy_blocks_kernel, dim3((unsigned)gx, (unsigned)gy), dim3(kCopyThreads), 0, stream,
                                  static_cast<uint4*>(pool), pairs, n, NB, blk_vec, dev_err);
    count_launch();
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "copy_blocks launch");
}

// One thread per table update (row, logical block, physical block); a negative row is padding.
__global__ void __launch_bounds__(256) update_tables_kernel(int32_t* __restrict__ tables, int N, int MB,
                                                            const int3* __restrict__ upd, int n, int* err) {
    griddep_wait();
    griddep_launch_dependents();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int3 u = upd[i];
    if (u.x < 0) return;
    if (u.x >= N || u.y < 0 || u.y >= MB) {
        flag_error(err, PA_DEV_ERR_BLOCK);
        return;
    }
    tables[(size_t)u.x * MB + u.y] = u.z;
}

pa_status launch_update_tables(int32_t* tables, int N, int MB, const int32_t* updates, int n, int* dev_err,
                               cudaStream_t stream) {
    if (n == 0) return PA_OK;
    cudaError_t e = launch_kernel(update_tables_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, tables, N, MB,
                                  reinterpret_cast<const int3*>(updates), n, dev_err);
    count_launch();
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "update_block_tables launch");
}

// Swap copy between two pools (either may be page-locked host memory): one CTA
// row per pair, grid.y chunks of the block, kCopyUnroll loads in flight per thread.
__global__ void __launch_bounds__(kCopyThreads) swap_blocks_kernel(uint4* __restrict__ dst,
                                                                   const uint4* __restrict__ src,
                                                                   const int64_t* __restrict__ pairs, int NB_dst,
                                                                   int NB_src, int64_t blk_vec, int* err) {
    griddep_wait();
    griddep_launch_dependents();
    const int i = blockIdx.x;
    const int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
    if (s < 0 || s >= NB_src || d < 0 || d >= NB_dst) {
        if (threadIdx.x == 0 && blockIdx.y == 0) flag_error(err, PA_DEV_ERR_BLOCK);
        return;
    }
    const uint4* sp = src + s * blk_vec;
    uint4* dp = dst + d * blk_vec;
    const int64_t chunk = (int64_t)kCopyThreads * kCopyUnroll;
    for (int64_t base = (int64_t)blockIdx.y * chunk; base < blk_vec; base += (int64_t)gridDim.y * chunk) {
        uint4 r[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t e = base + u * kCopyThreads + threadIdx.x;
            if (e < blk_vec) r[u] = sp[e];
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t e = base + u * kCopyThreads + threadIdx.x;
            if (e < blk_vec) dp[e] = r[u];
        }
    }
}

pa_status launch_swap_blocks(void* dst, int NB_dst, const void* src, int NB_src, const int64_t* pairs, int n,
                             int64_t blk_bytes, int* dev_err, cudaStream_t stream) {
    if (n == 0) return PA_OK;
    const int64_t blk_vec = blk_bytes / 16;
    const int64_t chunk = (int64_t)kCopyThreads * kCopyUnroll;
    int64_t gy = (blk_vec + chunk - 1) / chunk;
    if (gy > 65535) gy = 65535;
    cudaError_t e = launch_kernel(swap_blocks_kernel, dim3(n, (unsigned)gy), dim3(kCopyThreads), 0, stream,
                                  static_cast<uint4*>(dst), static_cast<const uint4*>(src), pairs, NB_dst, NB_src,
                                  blk_vec, dev_err);
    count_launch();
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "swap_blocks launch");
}

// Cache write for the contiguous per-request layout: token i's K and V rows go to
// request req_ids[i] at position positions[i] (offset (req * S + pos) rows).
__global__ void __launch_bounds__(128) write_contiguous_kernel(const uint4* __restrict__ k,
                                                               const uint4* __restrict__ v, uint4* __restrict__ kbuf,
                                                               uint4* __restrict__ vbuf,
                                                               const int32_t* __restrict__ req_ids,
                                                               const int32_t* __restrict__ pos, int T, int N_max,
                                                               int S, int row_vec, int* err) {
    griddep_wait();
    griddep_launch_dependents();
    for (int i = blockIdx.x; i < T; i += gridDim.x) {
        const int r = req_ids[i], t = pos[i];
        if (r < 0) continue;  // padding
        if (r >= N_max || t < 0 || t >= S) {
            if (threadIdx.x == 0) flag_error(err, r >= N_max ? PA_DEV_ERR_REQ : PA_DEV_ERR_SLOT);
            continue;
        }
        const int64_t row = ((int64_t)r * S + t) * row_vec;
        const uint4* sk = k + (int64_t)i * row_vec;
        const uint4* sv = v + (int64_t)i * row_vec;
        for (int e = threadIdx.x; e < row_vec; e += blockDim.x) {
            const uint4 a = sk[e];
            const uint4 b = sv[e];
            kbuf[row + e] = a;
            vbuf[row + e] = b;
        }
    }
}

pa_status launch_write_contiguous(const void* k, const void* v, void* k_buf, void* v_buf, const int32_t* req_ids,
                                  const int32_t* positions, int T, int N_max, int S, int H_kv, int D, int* dev_err,
                                  cudaStream_t stream) {
    if (T == 0) return PA_OK;
    const int row_vec = H_kv * D * 2 / 16;
    const int grid = token_grid(T);
    cudaError_t e = launch_kernel(write_contiguous_kernel, dim3(grid), dim3(128), 0, stream,
                                  static_cast<const uint4*>(k), static_cast<const uint4*>(v),
                                  static_cast<uint4*>(k_buf), static_cast<uint4*>(v_buf), req_ids, positions, T, N_max,
                                  S, row_vec, dev_err);
    count_launch();
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "write_contiguous launch");
}

}  // namespace pa

// decode.cu -- paged (and contiguous) decode attention for sm_103a.
//
// Method: PagedAttention explainer (0h-n0.github.io, arXiv 2309.06180),
// 技術的詳細 / PagedAttentionアルゴリズム (decode equation; K and V reached through
// the block table) and アルゴリズムの擬似コード (walk the blocks in order, keep a
// running maximum, exponential sum and rescaled output).  The contiguous variant
// follows the vAttention explainer (arXiv 2405.04437), 技術的詳細 /
// リクエスト単位のKVキャッシュインデキシング (request r at offset r * S).
//
// Three kernels per call:
//  1. plan_kernel (one CTA per slice of consecutive sequences): splits every
//     context into partitions of PT tokens and writes one work record (seq, kv
//     head, partition, ctx) per (partition, kv head) in longest-first order:
//     whole partitions in sequence order, then the ragged last partitions by
//     decreasing length.
//  2. attend_kernel (persistent, 4 CTAs per SM, 2 warps each): CTA c takes the
//     whole-partition records c, c + grid, ..., then ragged tails from a shared
//     counter, longest first; it computes record c from the lengths and streams
//     it while the schedule is still being written.  Warp 1 (producer) streams
//     each record's K/V through a ring of shared-memory stages with TMA: one
//     5-D tensor copy per KV block brings the block's K and V rows of one head,
//     128-byte swizzled;
//     the first stage of a record also carries the record's G query rows.
//     Warp 0 (consumer) computes S^T = K Q^T and O^T += V^T P^T with
//     mma.sync m16n8k16 (tokens on M, the <= 8 query heads of the KV head on N),
//     an online softmax in base 2 between stages, and writes the normalised
//     output, or the partition's (m2, l, acc) when the context has several
//     (stored with an L2 evict_last policy for the merge).
//  3. partition_reduce_kernel (one warp per row; partition_reduce_wide_kernel,
//     one CTA per row, from 32 partitions per row): merges the partials of
//     multi-partition rows.
// Each kernel is launched with programmatic stream serialisation, so its CTAs
// start while the previous kernel drains and wait (griddepcontrol.wait)
// before touching memory the previous kernel writes.
#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "pa_device.cuh"

namespace pa {

constexpr int kNumBins = 2048;
constexpr int kPlanThreads = 1024;
constexpr int kAttnThreads = 64;
constexpr int kEarlySeqs = 256;  // sequences a CTA scans for its first record before the schedule is written
constexpr uint32_t kSwzRowBytes = 128;

enum : int { kFirst = 1, kLast = 2, kDone = 4 };

struct __align__(16) StageMeta {
    int s, h, part, ctx;
    int tok0, n_valid, flags, pad;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Partition length for partition_tokens == 0: kDefaultPartition unless PA_DECODE_PARTITION names another
// multiple of the stage length (read once; a tuning knob like PA_DECODE_CTAS_PER_SM).
static int default_partition() {
    static const int pt = [] {
        const char* v = std::getenv("PA_DECODE_PARTITION");
        const int x = (v && *v) ? std::atoi(v) : 0;
        return x > 0 && x % kStageTok == 0 ? x : kDefaultPartition;
    }();
    return pt;
}

bool workspace_layout(int N, int H_q, int H_kv, int D, int max_ctx, int partition_tokens, WorkspaceLayout* L) {
    if (N <= 0 || H_q <= 0 || H_kv <= 0 || D <= 0 || max_ctx <= 0) return false;
    int PT;
    if (partition_tokens == 0)
        PT = default_partition();
    else if (partition_tokens == -1)
        PT = kUnpartitioned;
    else if (partition_tokens > 0 && partition_tokens % kStageTok == 0)
        PT = partition_tokens;
    else
        return false;
    const int P = PT >= kUnpartitioned ? 1 : (max_ctx + PT - 1) / PT;
    size_t off = 0;
    L->header = off;  // record count, tail counter, whole-partition record count
    off = align256(off + 16);
    L->nparts = off;
    off = align256(off + sizeof(int) * (size_t)N);
    L->records = off;
    off = align256(off + sizeof(int4) * (size_t)N * P * H_kv);
    const size_t rows = (size_t)N * H_q * P;
    if (P > 1) {
        L->part_m2 = off;
        off = align256(off + sizeof(float) * rows);
        L->part_l = off;
        off = align256(off + sizeof(float) * rows);
        L->part_acc = off;
        off = align256(off + sizeof(float) * rows * D);
    } else {
        L->part_m2 = L->part_l = L->part_acc = 0;
    }
    L->total = off;
    L->P = P;
    L->PT = PT;
    return true;
}

// ============================================================================= 1. schedule

__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Records for ragged last partitions are ordered by decreasing length through
// bins of kStageTok tokens (the top bin collects everything longer).
__device__ __forceinline__ int size_bin(int tokens, int nbins) {
    const int b = (tokens + kStageTok - 1) / kStageTok;
    return b < nbins ? b : nbins - 1;
}

static int plan_bins(int PT, int max_ctx) {
    const int longest_tail = PT >= kUnpartitioned ? max_ctx : PT - 1;
    const int n = (longest_tail + kStageTok - 1) / kStageTok + 1;
    return n < kNumBins ? n : kNumBins;
}

// The schedule is written by several CTAs.  CTA j owns the sequences [j*S, min(N, (j+1)*S)) and writes only their
// records, so the record stores of a call spread over the grid instead of queueing in one SM (a one-CTA schedule
// took about 16K cycles for the 7.9K records of 256 Llama-3-8B-shaped sequences).  To place its slice a CTA reads every
// context length: its first whole partition follows the whole partitions of all earlier sequences, and its
// ragged tails of one length bin follow that bin's tails from earlier slices.  Inside a CTA each warp writes whole
// sequences' records with its lanes on consecutive records, so a long sequence's P * H_kv records do not queue up
// behind one thread.  Within a (slice, bin) the tails' order is that of the atomic increments.
constexpr int kPlanSlice = 32;  // sequences per CTA while the grid still fits on the SMs

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* __restrict__ ctx_lens,
                                                                  const int32_t* __restrict__ req_ids, int N,
                                                                  int H_kv, int PT, int max_ctx, int cap, int N_max,
                                                                  int nbins, int* __restrict__ header,
                                                                  int4* __restrict__ rec, int* __restrict__ nparts,
                                                                  int* err) {
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int bins[kNumBins];       // tails per bin over all sequences, then this slice's next tail slot per bin
    __shared__ int before[kNumBins];     // tails per bin over the sequences before the slice
    __shared__ int pre[kPlanThreads];    // per sequence of a chunk: global index of its first whole partition
    __shared__ int cctx[kPlanThreads];   // per sequence of a chunk: checked context length (0: invalid)
    __shared__ int warp_sum[2][32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int S = (N + gridDim.x - 1) / gridDim.x;
    const int lo = min(N, (int)blockIdx.x * S), n = min(N, lo + S) - lo;
    for (int b = tid; b < nbins; b += blockDim.x) bins[b] = before[b] = 0;
    // context length of sequence s, 0 for an invalid length, -1 for an invalid request id
    auto checked_ctx = [&](int s) -> int {
        const int c = ctx_lens[s];
        if (c < 1 || c > max_ctx || c > cap) return 0;
        if (req_ids) {
            const int r = req_ids[s];
            if (r < 0 || r >= N_max) return -1;
        }
        return c;
    };
    __syncthreads();

    // pass 1 over every sequence: whole partitions in total and before the slice, tail histograms; the slice's
    // partition counts and error flags
    // (whole warps step together so that lanes of one bin add their count with one atomic)
    int full_all = 0, full_before = 0;
    for (int s0 = warp * 32; s0 < N; s0 += blockDim.x) {
        const int s = s0 + lane;
        const int c = s < N ? checked_ctx(s) : 0;
        const bool mine = s >= lo && s < lo + n;
        if (c <= 0 && mine) {
            flag_error(err, c == 0 ? PA_DEV_ERR_CTX : PA_DEV_ERR_REQ);
            nparts[s] = 0;
        }
        const int nf = c > 0 ? c / PT : 0, rem = c > 0 ? c - nf * PT : 0;
        full_all += nf;
        if (s < lo) full_before += nf;
        if (mine && c > 0) nparts[s] = nf + (rem > 0);
        const int b = rem > 0 ? size_bin(rem, nbins) : -1;
        const unsigned same = __match_any_sync(0xffffffffu, b);
        if (b >= 0 && lane == __ffs(same) - 1) atomicAdd(&bins[b], __popc(same));
        const int bb = s < lo ? b : -1;
        const unsigned same_before = __match_any_sync(0xffffffffu, bb);
        if (bb >= 0 && lane == __ffs(same_before) - 1) atomicAdd(&before[bb], __popc(same_before));
    }
    full_all = __reduce_add_sync(0xffffffffu, full_all);
    full_before = __reduce_add_sync(0xffffffffu, full_before);
    if (lane == 0) {
        warp_sum[0][warp] = full_all;
        warp_sum[1][warp] = full_before;
    }
    __syncthreads();
    if (warp == 0) {
        const int t = __reduce_add_sync(0xffffffffu, lane < nwarps ? warp_sum[0][lane] : 0);
        const int f = __reduce_add_sync(0xffffffffu, lane < nwarps ? warp_sum[1][lane] : 0);
        // descending exclusive scan of the tail histogram: longest tails first, after all whole partitions; the
        // slice's tails of a bin start after the earlier slices' tails of that bin
        const int chunk = (nbins + 31) / 32;
        int sum = 0;
        for (int j = lane * chunk; j < min(nbins, (lane + 1) * chunk); ++j) sum += bins[nbins - 1 - j];
        const int tincl = warp_incl_scan(sum);
        int run = t + tincl - sum;
        for (int j = lane * chunk; j < min(nbins, (lane + 1) * chunk); ++j) {
            const int b = nbins - 1 - j, c = bins[b];
            bins[b] = run + before[b];
            run += c;
        }
        if (lane == 31 && blockIdx.x == 0) {
            header[0] = (t + tincl) * H_kv;
            header[1] = 0;
            header[2] = t * H_kv;
        }
        if (lane == 0) warp_sum[1][0] = f;
    }
    __syncthreads();
    int base = warp_sum[1][0];  // whole partitions before the current chunk of the slice

    // pass 2 over the slice, blockDim.x sequences at a time: an exclusive scan gives each sequence the index of its
    // first whole partition, then each warp writes whole sequences' records (one per (partition, kv head))
    for (int c0 = 0; c0 < n; c0 += blockDim.x) {
        const int m = min((int)blockDim.x, n - c0);
        int c = tid < m ? checked_ctx(lo + c0 + tid) : 0;
        c = c > 0 ? c : 0;
        if (tid < m) cctx[tid] = c;
        const int v = c / PT;
        const int incl = warp_incl_scan(v);
        __syncthreads();
        if (lane == 31) warp_sum[0][warp] = incl;
        __syncthreads();
        if (warp == 0) warp_sum[0][lane] = warp_incl_scan(lane < nwarps ? warp_sum[0][lane] : 0);
        __syncthreads();
        if (tid < m) pre[tid] = base + incl - v + (warp ? warp_sum[0][warp - 1] : 0);
        base += warp_sum[0][nwarps - 1];
        __syncthreads();
        for (int i = warp; i < m; i += nwarps) {
            const int ci = cctx[i];
            if (ci == 0) continue;
            const int s = lo + c0 + i, nf = ci / PT, rem = ci - nf * PT;
            int4* r0 = rec + (size_t)pre[i] * H_kv;
            for (int k = lane; k < nf * H_kv; k += 32) r0[k] = make_int4(s, k % H_kv, k / H_kv, ci);
            if (rem > 0) {
                int pos = 0;
                if (lane == 0) pos = atomicAdd(&bins[size_bin(rem, nbins)], 1);
                pos = __shfl_sync(0xffffffffu, pos, 0);
                for (int h = lane; h < H_kv; h += 32) rec[(size_t)pos * H_kv + h] = make_int4(s, h, nf, ci);
            }
        }
        __syncthreads();
    }
}

// ============================================================================= merge of partition partials

template <typename OutT, int D>
__device__ __forceinline__ void store_row(OutT* dst, const float (&o)[D / 32]) {
    constexpr int V = D / 32;
    const int lane = threadIdx.x & 31;
    if constexpr (sizeof(OutT) == 4 && V == 4) {
        *reinterpret_cast<float4*>(dst + lane * V) = make_float4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
        for (int v = 0; v < V; ++v) dst[lane * V + v] = from_float<OutT>(o[v]);
    }
}

// ============================================================================= 2. attention

struct AttnParams {
    const int4* rec;
    int* header;
    const int32_t* tables;
    int MB, B, NB;
    const int32_t* req_ids;
    int S_max;
    const void* q;
    int H_q, G;
    void* out;
    int out_dtype;
    float* part_m2;
    float* part_l;
    float* part_acc;
    int P, PT;
    // inputs of the schedule, for a CTA that starts on its first record before the schedule is written
    const int32_t* ctx_lens;
    int N, H_kv, max_ctx, cap, N_max;
    float scale_log2;
    int nstage;
    uint64_t wait_ns;  // limit of the ring waits (the exit path waits with kWaitLimitNs)
    int* err;
};

template <int D>
struct Geo {
    static constexpr int DH = D / 64;                               // 128-byte rows per head row
    static constexpr uint32_t kStageBytes = kStageTok * D * 2 * 2;  // K and V of one stage
    static constexpr uint32_t kQBytes = kMaxGroup * D * 2;          // the record's query rows
    static constexpr uint32_t kSlotBytes = kStageBytes + kQBytes;   // a multiple of 1024
    static constexpr int kSub = kStageTok / 16;                     // 16-token mma tiles per stage
    static_assert(kSlotBytes % 1024 == 0, "slots keep the 1024-byte swizzle alignment");
};

template <int D>
static size_t attend_smem_bytes(int nstage) {
    return 1024 + (size_t)nstage * (Geo<D>::kSlotBytes + sizeof(StageMeta) + 16) + 16;
}

template <typename T, int D, bool PAGED>
__global__ void __launch_bounds__(kAttnThreads) attend_kernel(const __grid_constant__ CUtensorMap tm_a,
                                                              const __grid_constant__ CUtensorMap tm_b,
                                                              const AttnParams p) {
    using G_ = Geo<D>;
    constexpr int DH = G_::DH;
    constexpr int NSUB = G_::kSub;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int nstage = p.nstage;
    StageMeta* meta = reinterpret_cast<StageMeta*>(base + (size_t)nstage * G_::kSlotBytes);
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(meta + nstage);
    uint64_t* empty_bar = full_bar + nstage;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty_bar + nstage);
    const uint32_t slots_s = smem_addr(base);
    const uint32_t full_s = smem_addr(full_bar), empty_s = smem_addr(empty_bar);

    if (threadIdx.x == 0) {
        for (int i = 0; i < nstage; ++i) {
            mbar_init(full_s + 8 * i, 1);
            mbar_init(empty_s + 8 * i, 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (threadIdx.x == 32) {
        prefetch_tmap(&tm_a);
        if (!PAGED) prefetch_tmap(&tm_b);
    }
    __syncthreads();
    // Everything up to the producer's join_schedule() overlaps the schedule kernel.  This kernel is only ever
    // launched right after the schedule kernel, whose CTAs let it start only once every kernel before them has
    // finished: from here on the call's inputs (lengths, tables, q, pool) are final, and the outputs and partials
    // this kernel writes are touched by no earlier kernel still running.  Only the schedule's own output (header,
    // records) needs the wait.
    griddep_launch_dependents();

    const int lane = threadIdx.x & 31;
    const int Beff = PAGED ? p.B : kStageTok;  // tokens per TMA box along the token axis
    const uint32_t blk_bytes = (uint32_t)Beff * D * 4;

    if (threadIdx.x >= 32) {
        // ------------------------------------------------------------------ producer warp
        int total = 0, nwhole = 0;
        bool joined = false;
        auto join_schedule = [&]() {
            griddep_wait();
            total = p.header[0];
            nwhole = p.header[2];
            joined = true;
        };
        const uint64_t pol = policy_evict_first();
        const int bps = kStageTok / Beff;  // boxes per stage
        int slot = 0;
        uint32_t ephase = 0;
        int narm = 0;  // stages armed so far (stage i's k-th arm completes phase k of full_bar[i])
        bool ok = true;
        const int4 none = make_int4(-1, 0, 0, 0);
        // record order: the whole partitions round robin (CTA c takes c, c + grid, ... below nwhole), then the
        // ragged tails from a shared counter, so the CTAs that run out of whole partitions first take the
        // longest tails; lane 0 asks for the index after the next record while the current one streams
        auto after = [&](int i) -> int {
            const int j = i + (int)gridDim.x;
            return j < nwhole ? j : nwhole + atomicAdd(p.header + 1, 1);
        };
        // The CTA's first record, whole partition blockIdx.x of the round robin, follows from the lengths alone
        // (the schedule orders whole partitions by sequence, partition, kv head): when it lies in the first
        // kEarlySeqs sequences the CTA streams it before the schedule is written, and joins the schedule for
        // the records after it.
        auto early_record = [&]() -> int4 {
            if (p.PT >= kUnpartitioned) return none;
            const int j = (int)blockIdx.x / p.H_kv, h = (int)blockIdx.x % p.H_kv;  // whole partition, kv head
            int c[kEarlySeqs / 32];
#pragma unroll
            for (int k = 0; k < kEarlySeqs / 32; ++k) {
                const int sq = 32 * k + lane;
                int v = sq < p.N ? p.ctx_lens[sq] : 0;
                if (v < 1 || v > p.max_ctx || v > p.cap) v = 0;  // as the schedule: no records
                if (!PAGED && v > 0) {
                    const int r = p.req_ids[sq];
                    if (r < 0 || r >= p.N_max) v = 0;
                }
                c[k] = v;
            }
            int run = 0;  // whole partitions of the sequences before chunk k
#pragma unroll
            for (int k = 0; k < kEarlySeqs / 32; ++k) {
                const int nf = c[k] / p.PT;
                const int incl = warp_incl_scan(nf);
                const unsigned hit = __ballot_sync(0xffffffffu, run + incl - nf <= j && j < run + incl);
                if (hit) {
                    const int src = __ffs(hit) - 1;
                    const int first = __shfl_sync(0xffffffffu, run + incl - nf, src);
                    return make_int4(32 * k + src, h, j - first, __shfl_sync(0xffffffffu, c[k], src));
                }
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            return none;
        };
        int4 cur = early_record(), nxt = none;
        int nidx = 0, pend = 0;
        // joins the schedule after the early first record: the record after it and the one after that
        auto join_after_first = [&]() {
            join_schedule();
            if (lane == 0) nidx = after((int)blockIdx.x);
            nidx = __shfl_sync(0xffffffffu, nidx, 0);
            nxt = nidx < total ? p.rec[nidx] : none;
            if (lane == 0 && nxt.x >= 0) pend = after(nidx);
        };
        if (cur.x < 0) {
            join_schedule();
            if (lane == 0) nidx = after((int)blockIdx.x - (int)gridDim.x);
            nidx = __shfl_sync(0xffffffffu, nidx, 0);
            cur = nidx < total ? p.rec[nidx] : none;
            if (lane == 0) nidx = after(nidx);
            nidx = __shfl_sync(0xffffffffu, nidx, 0);
            nxt = nidx < total ? p.rec[nidx] : none;
            if (lane == 0 && nxt.x >= 0) pend = after(nidx);
        }
        // table entries of the first 32 boxes of `it` starting at box `cb`
        auto load_entries = [&](const int4& it, int cb) -> int {
            const int t0 = it.z * p.PT;
            const int ntok = min(p.PT, it.w - t0);
            const int nblk = (ntok + Beff - 1) / Beff;
            const int b = cb + lane;
            if (PAGED) return b < nblk ? p.tables[(size_t)it.x * p.MB + t0 / Beff + b] : 0;
            return p.req_ids[it.x];
        };
        int ent = cur.x >= 0 ? load_entries(cur, 0) : 0;
        while (cur.x >= 0 && ok) {
            const int s = cur.x, h = cur.y, part = cur.z, ctx = cur.w;
            const int t0 = part * p.PT;
            const int ntok = min(p.PT, ctx - t0);
            const int nblk = (ntok + Beff - 1) / Beff;
            const int nst = (ntok + kStageTok - 1) / kStageTok;
            int st = 0;
            for (int cb = 0; cb < nblk && ok; cb += 32) {
                int ent_nx = 0;
                if (cb + 32 < nblk)
                    ent_nx = load_entries(cur, cb + 32);
                else if (joined && nxt.x >= 0)
                    ent_nx = load_entries(nxt, 0);
                const int cend = min(cb + 32, nblk);
                for (int b0 = cb; b0 < cend; b0 += bps, ++st) {
                    if (!joined && st == nstage) {
                        // the ring is full of the early record: learn the next one while it drains
                        join_after_first();
                        if (cb + 32 >= nblk && nxt.x >= 0) ent_nx = load_entries(nxt, 0);
                    }
                    if (lane == 0) ok = mbar_wait_bounded(empty_s + 8 * slot, ephase ^ 1, abort_flag, p.wait_ns);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    ++narm;  // armed below: expect_tx and every copy of the stage, with no wait in between
                    const int tok0 = st * kStageTok;
                    const int nvalid = min(kStageTok, ntok - tok0);
                    const int nb = min(bps, nblk - b0);
                    const bool first = st == 0, last = st == nst - 1;
                    const uint32_t kv_s = slots_s + (uint32_t)slot * G_::kSlotBytes;
                    const uint32_t bar = full_s + 8 * slot;
                    if (lane == 0) {
                        StageMeta m;
                        m.s = s;
                        m.h = h;
                        m.part = part;
                        m.ctx = ctx;
                        m.tok0 = t0 + tok0;
                        m.n_valid = nvalid;
                        m.flags = (first ? kFirst : 0) | (last ? kLast : 0);
                        m.pad = 0;
                        meta[slot] = m;
                        uint32_t bytes = PAGED ? (uint32_t)nb * blk_bytes : G_::kStageBytes;
                        if (first) bytes += (uint32_t)p.G * D * 2;
                        mbar_arrive_expect_tx(bar, bytes);
                        if (first) {
                            const T* qsrc = static_cast<const T*>(p.q) + ((size_t)s * p.H_q + (size_t)h * p.G) * D;
                            bulk_load(kv_s + G_::kStageBytes, qsrc, (uint32_t)p.G * D * 2, bar);
                        }
                    }
                    if (PAGED) {
                        for (int b = 0; b < bps; ++b) {
                            int e = __shfl_sync(0xffffffffu, ent, (b0 - cb + b) & 31);
                            if (lane == 0 && b < nb) {
                                if ((unsigned)e >= (unsigned)p.NB) {
                                    flag_error(p.err, PA_DEV_ERR_BLOCK);
                                    e = p.NB;  // past the tensor: TMA fills zeros
                                }
                                tma_load_5d(kv_s + (uint32_t)b * blk_bytes, &tm_a, bar, 0, e * p.B, 0, h, 0, pol);
                            }
                        }
                    } else if (lane == 0) {
                        const int row = ent * p.S_max + t0 + tok0;
                        tma_load_4d(kv_s, &tm_a, bar, 0, row, 0, h, pol);
                        tma_load_4d(kv_s + G_::kStageBytes / 2, &tm_b, bar, 0, row, 0, h, pol);
                    }
                    if (++slot == nstage) {
                        slot = 0;
                        ephase ^= 1;
                    }
                }
                ent = ent_nx;
            }
            if (!joined) {
                // an early first record shorter than the ring: the records after it come from the schedule
                join_after_first();
                ent = nxt.x >= 0 ? load_entries(nxt, 0) : 0;
            }
            cur = nxt;
            nidx = __shfl_sync(0xffffffffu, pend, 0);
            nxt = nidx < total ? p.rec[nidx] : none;
            if (lane == 0 && nxt.x >= 0) pend = after(nidx);
        }
        if (ok && lane == 0) {
            ok = mbar_wait_bounded(empty_s + 8 * slot, ephase ^ 1, abort_flag, p.wait_ns);
            if (ok) {
                meta[slot].flags = kDone;
                mbar_arrive(full_s + 8 * slot);
                ++narm;
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (lane == 0) {
            if (!ok) {
                flag_error(p.err, PA_DEV_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            // Copies land in this CTA's shared memory, so it may not exit while one is in flight.  When the
            // consumer gave up (a wait ran out, or it saw the abort flag), stages it never reached can still be
            // landing, whether or not this warp itself ran into a wait.  Stage i's last arm is arm
            // i + m * nstage, m = (narm - 1 - i) / nstage, and it completes phase m of full_bar[i]; waiting on
            // that phase's parity covers every earlier arm too (each was consumed before the next was armed).
            // In a call that ran to completion every such phase is already complete.
            for (int i = 0; i < nstage && i < narm; ++i) {
                const int m = (narm - 1 - i) / nstage;
                mbar_wait_bounded(full_s + 8 * i, (uint32_t)(m & 1), nullptr, kWaitLimitNs);
            }
        }
        return;
    }

    // ---------------------------------------------------------------------- consumer warp
    const int g4 = lane >> 2, t4 = lane & 3;
    const int lgB = 31 - __clz(Beff);
    // ldmatrix row addresses (relative to a slot) and swizzle masks, per 16-token tile j and 64-column half dh
    uint32_t kofs[NSUB][DH], kx[NSUB][DH], vofs[NSUB][DH], vx[NSUB][DH];
    {
        const int k_tok = (lane & 7) + ((lane >> 3) & 1) * 8, k_hi = lane >> 4;
        const int v_tok = (lane & 7) + ((lane >> 4) & 1) * 8, v_hi = (lane >> 3) & 1;
#pragma unroll
        for (int j = 0; j < NSUB; ++j) {
#pragma unroll
            for (int dh = 0; dh < DH; ++dh) {
                int tok = 16 * j + k_tok;
                int row = (tok >> lgB) * (2 * DH * Beff) + dh * Beff + (tok & (Beff - 1));
                kofs[j][dh] = (uint32_t)row * kSwzRowBytes;
                kx[j][dh] = (uint32_t)((k_hi ^ (row & 7)) << 4);
                tok = 16 * j + v_tok;
                row = (tok >> lgB) * (2 * DH * Beff) + (DH + dh) * Beff + (tok & (Beff - 1));
                vofs[j][dh] = (uint32_t)row * kSwzRowBytes;
                vx[j][dh] = (uint32_t)((v_hi ^ (row & 7)) << 4);
            }
        }
    }
    constexpr int NT = D / 16;
    float O[NT][4];
    uint32_t qf[NT][2];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int slot = 0;
    uint32_t fphase = 0;
    const float NEG_INF = -INFINITY;
    while (true) {
        if (!mbar_wait_bounded(full_s + 8 * slot, fphase, abort_flag, p.wait_ns)) {
            if (lane == 0) {
                flag_error(p.err, PA_DEV_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            break;
        }
        const StageMeta mt = meta[slot];
        if (mt.flags & kDone) break;
        const uint32_t kv_s = slots_s + (uint32_t)slot * G_::kSlotBytes;
        const uint8_t* kv_g = base + (size_t)slot * G_::kSlotBytes;
        if (mt.flags & kFirst) {
            const uint8_t* qs = kv_g + G_::kStageBytes;
#pragma unroll
            for (int ks = 0; ks < NT; ++ks) {
                const int d = 16 * ks + 2 * t4;
                qf[ks][0] = g4 < p.G ? *reinterpret_cast<const uint32_t*>(qs + ((size_t)g4 * D + d) * 2) : 0u;
                qf[ks][1] = g4 < p.G ? *reinterpret_cast<const uint32_t*>(qs + ((size_t)g4 * D + d + 8) * 2) : 0u;
            }
#pragma unroll
            for (int i = 0; i < NT; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
            m0 = m1 = NEG_INF;
            l0 = l1 = 0.f;
        }
        const int nvalid = mt.n_valid;

        // S^T = K Q^T for each 16-token tile (two accumulators to shorten the dependency chain)
        float sc[NSUB][4];
#pragma unroll
        for (int j = 0; j < NSUB; ++j) {
            sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
            if (16 * j < nvalid) {
                float a[4] = {0.f, 0.f, 0.f, 0.f}, b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < NT; ++ks) {
                    const int dh = ks >> 2;
                    const uint32_t addr = kv_s + kofs[j][dh] + ((uint32_t)(((ks & 3) * 2) << 4) ^ kx[j][dh]);
                    uint32_t r0, r1, r2, r3;
                    ldmatrix_x4(addr, r0, r1, r2, r3);
                    if (ks & 1)
                        Mma<T>::run(b, r0, r1, r2, r3, qf[ks][0], qf[ks][1]);
                    else
                        Mma<T>::run(a, r0, r1, r2, r3, qf[ks][0], qf[ks][1]);
                }
#pragma unroll
                for (int r = 0; r < 4; ++r) sc[j][r] = a[r] + b[r];
            }
        }
        // scale to base 2, mask tokens past the context, stage maximum per head
        float x0 = NEG_INF, x1 = NEG_INF;
#pragma unroll
        for (int j = 0; j < NSUB; ++j) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int tok = 16 * j + g4 + (r >> 1) * 8;
                sc[j][r] = tok < nvalid ? sc[j][r] * p.scale_log2 : NEG_INF;
            }
            x0 = fmaxf(x0, fmaxf(sc[j][0], sc[j][2]));
            x1 = fmaxf(x1, fmaxf(sc[j][1], sc[j][3]));
        }
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, o));
            x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, o));
        }
        const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
        const float a0 = fast_exp2(m0 - n0), a1 = fast_exp2(m1 - n1);
        m0 = n0;
        m1 = n1;
        if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                O[i][0] *= a0;
                O[i][1] *= a1;
                O[i][2] *= a0;
                O[i][3] *= a1;
            }
            l0 *= a0;
            l1 *= a1;
        }
        // probabilities as a high and a low 16-bit part, transposed into mma B fragments
        uint32_t bh[NSUB][2], bl[NSUB][2];
#pragma unroll
        for (int j = 0; j < NSUB; ++j) {
            const float p0 = fast_exp2(sc[j][0] - n0), p1 = fast_exp2(sc[j][1] - n1);
            const float p2 = fast_exp2(sc[j][2] - n0), p3 = fast_exp2(sc[j][3] - n1);
            l0 += p0 + p2;
            l1 += p1 + p3;
            const uint32_t h01 = Mma<T>::pack(p0, p1), h23 = Mma<T>::pack(p2, p3);
            const float2 f01 = Mma<T>::unpack(h01), f23 = Mma<T>::unpack(h23);
            const uint32_t lo01 = Mma<T>::pack(p0 - f01.x, p1 - f01.y), lo23 = Mma<T>::pack(p2 - f23.x, p3 - f23.y);
            bh[j][0] = movmatrix_trans(h01);
            bh[j][1] = movmatrix_trans(h23);
            bl[j][0] = movmatrix_trans(lo01);
            bl[j][1] = movmatrix_trans(lo23);
        }
        // V rows past the context inside the last tile may hold anything (even NaN); zero them
        if (nvalid & 15) {
            const int t_lo = nvalid, t_hi = (nvalid + 15) & ~15;
            const int nchunk = (t_hi - t_lo) * DH * 8;
            for (int c = lane; c < nchunk; c += 32) {
                const int tok = t_lo + c / (DH * 8);
                const int rem = c % (DH * 8);
                const int dh = rem >> 3, ch = rem & 7;
                const int row = (tok >> lgB) * (2 * DH * Beff) + (DH + dh) * Beff + (tok & (Beff - 1));
                const uint32_t a = kv_s + (uint32_t)row * kSwzRowBytes + (uint32_t)ch * 16;
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
        }
        // O^T += V^T P^T
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            const int dh = i >> 2;
#pragma unroll
            for (int j = 0; j < NSUB; ++j) {
                if (16 * j < nvalid) {
                    const uint32_t addr = kv_s + vofs[j][dh] + ((uint32_t)(((i & 3) * 2) << 4) ^ vx[j][dh]);
                    uint32_t r0, r1, r2, r3;
                    ldmatrix_x4_trans(addr, r0, r1, r2, r3);
                    Mma<T>::run(O[i], r0, r1, r2, r3, bh[j][0], bh[j][1]);
                    Mma<T>::run(O[i], r0, r1, r2, r3, bl[j][0], bl[j][1]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_s + 8 * slot);

        if (mt.flags & kLast) {
            float L0 = l0, L1 = l1;
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                L0 += __shfl_xor_sync(0xffffffffu, L0, o);
                L1 += __shfl_xor_sync(0xffffffffu, L1, o);
            }
            const int np = p.PT >= kUnpartitioned ? 1 : (mt.ctx + p.PT - 1) / p.PT;
            const int h0 = 2 * t4, h1 = h0 + 1;
            const size_t qrow0 = (size_t)mt.s * p.H_q + (size_t)mt.h * p.G;
            if (np == 1) {
                const float i0 = 1.f / L0, i1 = 1.f / L1;
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    const int d = 16 * i + g4;
                    if (h0 < p.G) {
                        const size_t o = (qrow0 + h0) * D + d;
                        if (p.out_dtype == PA_F32) {
                            static_cast<float*>(p.out)[o] = O[i][0] * i0;
                            static_cast<float*>(p.out)[o + 8] = O[i][2] * i0;
                        } else {
                            static_cast<T*>(p.out)[o] = from_float<T>(O[i][0] * i0);
                            static_cast<T*>(p.out)[o + 8] = from_float<T>(O[i][2] * i0);
                        }
                    }
                    if (h1 < p.G) {
                        const size_t o = (qrow0 + h1) * D + d;
                        if (p.out_dtype == PA_F32) {
                            static_cast<float*>(p.out)[o] = O[i][1] * i1;
                            static_cast<float*>(p.out)[o + 8] = O[i][3] * i1;
                        } else {
                            static_cast<T*>(p.out)[o] = from_float<T>(O[i][1] * i1);
                            static_cast<T*>(p.out)[o + 8] = from_float<T>(O[i][3] * i1);
                        }
                    }
                }
            } else {
                const size_t r0 = (qrow0 + h0) * p.P + mt.part, r1 = (qrow0 + h1) * p.P + mt.part;
                // the merge reads the partials right after this kernel: keep them in L2
                const uint64_t keep = policy_evict_last();
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    const int d = 16 * i + g4;
                    if (h0 < p.G) {
                        st_hint(p.part_acc + r0 * D + d, O[i][0], keep);
                        st_hint(p.part_acc + r0 * D + d + 8, O[i][2], keep);
                    }
                    if (h1 < p.G) {
                        st_hint(p.part_acc + r1 * D + d, O[i][1], keep);
                        st_hint(p.part_acc + r1 * D + d + 8, O[i][3], keep);
                    }
                }
                if (g4 == 0) {
                    if (h0 < p.G) {
                        st_hint(p.part_m2 + r0, m0, keep);
                        st_hint(p.part_l + r0, L0, keep);
                    }
                    if (h1 < p.G) {
                        st_hint(p.part_m2 + r1, m1, keep);
                        st_hint(p.part_l + r1, L1, keep);
                    }
                }
            }
        }
        if (++slot == nstage) {
            slot = 0;
            fphase ^= 1;
        }
    }
}

// ============================================================================= 3. partition merge

// One warp per output row, 8 rows per CTA, so the whole merge is one wave of
// short-lived warps.  The merge is latency bound (its inputs sit in L2), so a
// warp issues every load of up to kMergeChunk partitions -- lane j's m2 and l
// of partition j, and each lane's D/32 columns of every partition's acc --
// before it uses any of them: one L2 round trip after the partition count
// instead of one per dependent step.  Longer rows take further chunks, the
// running maximum and sums rescaled between chunks.
constexpr int kReduceWarps = 8;
constexpr int kMergeChunk = 8;

template <typename OutT, int D>
__global__ void __launch_bounds__(kReduceWarps * 32) partition_reduce_kernel(
    OutT* __restrict__ out, const float* __restrict__ m2, const float* __restrict__ l, const float* __restrict__ acc,
    const int32_t* __restrict__ nparts, int rows_per_seq, int R, int P, int skip_single, int* err) {
    constexpr int V = D / 32;
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kReduceWarps + (threadIdx.x >> 5);
    if (r >= R) return;
    const int np = nparts[r / rows_per_seq];
    if (skip_single && np <= 1) return;  // written by the attention kernel, or an invalid sequence
    if (np < 1 || np > P) {
        if (lane == 0) flag_error(err, PA_DEV_ERR_CTX);
        return;
    }
    const float* mr = m2 + (size_t)r * P;
    const float* lr = l + (size_t)r * P;
    const float* ar = acc + (size_t)r * P * D + lane * V;
    float M = -INFINITY, den = 0.f, o[V];
#pragma unroll
    for (int v = 0; v < V; ++v) o[v] = 0.f;
    for (int base = 0; base < np; base += kMergeChunk) {
        const int n = min(kMergeChunk, np - base);
        // every load of the chunk first
        const float mv = lane < n ? mr[base + lane] : -INFINITY;
        const float lv = lane < n ? lr[base + lane] : 0.f;
        float a[kMergeChunk][V];
#pragma unroll
        for (int j = 0; j < kMergeChunk; ++j) {
            if (j < n) {
                const float* src = ar + (size_t)(base + j) * D;
                if constexpr (V == 4) {
                    const float4 x = *reinterpret_cast<const float4*>(src);
                    a[j][0] = x.x;
                    a[j][1] = x.y;
                    a[j][2] = x.z;
                    a[j][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2*>(src);
                    a[j][0] = x.x;
                    a[j][1] = x.y;
                }
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) a[j][v] = 0.f;
            }
        }
        float mc = mv;
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, k));
        const float Mn = fmaxf(M, mc);  // finite: every partition holds at least one token
        const float f = fast_exp2(M - Mn);  // 0 on the first chunk (M = -inf)
        den *= f;
#pragma unroll
        for (int v = 0; v < V; ++v) o[v] *= f;
        M = Mn;
        const float w = lane < n ? fast_exp2(mv - Mn) : 0.f;
        den += w * lv;
#pragma unroll
        for (int j = 0; j < kMergeChunk; ++j) {
            const float wj = __shfl_sync(0xffffffffu, w, j);
#pragma unroll
            for (int v = 0; v < V; ++v) o[v] += wj * a[j][v];
        }
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) den += __shfl_xor_sync(0xffffffffu, den, k);
    const float inv = 1.f / den;
#pragma unroll
    for (int v = 0; v < V; ++v) o[v] *= inv;
    store_row<OutT, D>(out + (size_t)r * D, o);
}

// Rows with many partitions (long contexts): one CTA per row, warp k merging partitions k, k + 8, ... and
// warp 0 combining the eight partial results, so no warp walks more than P / 8 partitions.
template <typename OutT, int D>
__global__ void __launch_bounds__(kReduceWarps * 32) partition_reduce_wide_kernel(
    OutT* __restrict__ out, const float* __restrict__ m2, const float* __restrict__ l, const float* __restrict__ acc,
    const int32_t* __restrict__ nparts, int rows_per_seq, int R, int P, int skip_single, int* err) {
    constexpr int V = D / 32;
    griddep_wait();
    griddep_launch_dependents();
    __shared__ float sM[kReduceWarps], sDen[kReduceWarps];
    __shared__ __align__(16) float sO[kReduceWarps][D];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int r = blockIdx.x;
    const int np = nparts[r / rows_per_seq];
    if (skip_single && np <= 1) return;  // uniform per CTA
    if (np < 1 || np > P) {
        if (threadIdx.x == 0) flag_error(err, PA_DEV_ERR_CTX);
        return;
    }
    const float* mr = m2 + (size_t)r * P;
    const float* lr = l + (size_t)r * P;
    const float* ar = acc + (size_t)r * P * D + lane * V;
    const int mine_n = np > warp ? (np - warp + kReduceWarps - 1) / kReduceWarps : 0;  // partitions of this warp
    // as the one-warp merge: every load of up to kMergeChunk of this warp's partitions first, then the sums
    float M = -INFINITY, den = 0.f, o[V];
#pragma unroll
    for (int v = 0; v < V; ++v) o[v] = 0.f;
    for (int base = 0; base < mine_n; base += kMergeChunk) {
        const int n = min(kMergeChunk, mine_n - base);
        const int pl = warp + kReduceWarps * (base + lane);
        const float mv = lane < n ? mr[pl] : -INFINITY;
        const float lv = lane < n ? lr[pl] : 0.f;
        float a[kMergeChunk][V];
#pragma unroll
        for (int j = 0; j < kMergeChunk; ++j) {
            const float* src = ar + (size_t)(warp + kReduceWarps * (base + j)) * D;
            if (j < n) {
                if constexpr (V == 4) {
                    const float4 x = *reinterpret_cast<const float4*>(src);
                    a[j][0] = x.x;
                    a[j][1] = x.y;
                    a[j][2] = x.z;
                    a[j][3] = x.w;
                } else {
                    const float2 x = *reinterpret_cast<const float2*>(src);
                    a[j][0] = x.x;
                    a[j][1] = x.y;
                }
            } else {
#pragma unroll
                for (int v = 0; v < V; ++v) a[j][v] = 0.f;
            }
        }
        float mc = mv;
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, k));
        const float Mn = fmaxf(M, mc);
        const float f = fast_exp2(M - Mn);  // 0 on the first chunk (M = -inf)
        den *= f;
#pragma unroll
        for (int v = 0; v < V; ++v) o[v] *= f;
        M = Mn;
        const float w = lane < n ? fast_exp2(mv - Mn) : 0.f;
        den += w * lv;
#pragma unroll
        for (int j = 0; j < kMergeChunk; ++j) {
            const float wj = __shfl_sync(0xffffffffu, w, j);
#pragma unroll
            for (int v = 0; v < V; ++v) o[v] += wj * a[j][v];
        }
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) den += __shfl_xor_sync(0xffffffffu, den, k);
    if (lane == 0) {
        sM[warp] = M;
        sDen[warp] = den;
    }
#pragma unroll
    for (int v = 0; v < V; ++v) sO[warp][lane * V + v] = o[v];
    __syncthreads();
    if (warp == 0) {
        float Mt = -INFINITY;
#pragma unroll
        for (int k = 0; k < kReduceWarps; ++k) Mt = fmaxf(Mt, sM[k]);
        float ot[V], dt = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) ot[v] = 0.f;
#pragma unroll
        for (int k = 0; k < kReduceWarps; ++k) {
            if (sM[k] == -INFINITY) continue;  // a warp without partitions
            const float f = fast_exp2(sM[k] - Mt);
            dt += f * sDen[k];
#pragma unroll
            for (int v = 0; v < V; ++v) ot[v] += f * sO[k][lane * V + v];
        }
        const float inv = 1.f / dt;
#pragma unroll
        for (int v = 0; v < V; ++v) ot[v] *= inv;
        store_row<OutT, D>(out + (size_t)r * D, ot);
    }
}

// Merges of at least this many partitions per row (the stride P) use one CTA per row: at P = 17 (Llama-3-8B
// decode, most rows 2-16 partitions) CTA-per-row cost 3 % of the step, at P = 64 (8 x 32K) it saved 9 %.
constexpr int kWideMergeParts = 32;

template <typename OutT>
static cudaError_t reduce_dispatch_d(void* out, const float* m2, const float* l, const float* acc,
                                     const int32_t* nparts, int rows_per_seq, int R, int P, int D, bool skip,
                                     int* err, cudaStream_t st) {
    const dim3 block(kReduceWarps * 32);
    if (P >= kWideMergeParts) {
        if (D == 128)
            return launch_kernel(partition_reduce_wide_kernel<OutT, 128>, dim3(R), block, 0, st,
                                 static_cast<OutT*>(out), m2, l, acc, nparts, rows_per_seq, R, P, skip ? 1 : 0, err);
        return launch_kernel(partition_reduce_wide_kernel<OutT, 64>, dim3(R), block, 0, st, static_cast<OutT*>(out), m2,
                             l, acc, nparts, rows_per_seq, R, P, skip ? 1 : 0, err);
    }
    const dim3 grid((R + kReduceWarps - 1) / kReduceWarps);
    if (D == 128)
        return launch_kernel(partition_reduce_kernel<OutT, 128>, grid, block, 0, st, static_cast<OutT*>(out), m2, l,
                             acc, nparts, rows_per_seq, R, P, skip ? 1 : 0, err);
    return launch_kernel(partition_reduce_kernel<OutT, 64>, grid, block, 0, st, static_cast<OutT*>(out), m2, l, acc,
                         nparts, rows_per_seq, R, P, skip ? 1 : 0, err);
}

pa_status launch_partition_reduce(void* out, int out_dtype, const float* m2, const float* l, const float* acc,
                                  const int32_t* nparts, int rows_per_seq, int R, int P, int D, bool skip_single,
                                  int* dev_err, cudaStream_t stream) {
    if (R == 0) return PA_OK;
    cudaError_t e;
    if (out_dtype == PA_F32)
        e = reduce_dispatch_d<float>(out, m2, l, acc, nparts, rows_per_seq, R, P, D, skip_single, dev_err, stream);
    else if (out_dtype == PA_F16)
        e = reduce_dispatch_d<__half>(out, m2, l, acc, nparts, rows_per_seq, R, P, D, skip_single, dev_err, stream);
    else
        e = reduce_dispatch_d<__nv_bfloat16>(out, m2, l, acc, nparts, rows_per_seq, R, P, D, skip_single, dev_err,
                                             stream);
    count_launch();
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "partition_reduce launch");
}

// ============================================================================= host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

static pa_status encode(CUtensorMap* m, int kv_dtype, int rank, const void* base, const cuuint64_t* dims,
                        const cuuint64_t* strides, const cuuint32_t* box) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, kv_dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return PA_OK;
}

static int env_int(const char* name, int dflt) {
    const char* s = std::getenv(name);
    if (!s || !*s) return dflt;
    return std::atoi(s);
}

template <typename T, int D, bool PAGED>
static pa_status run_attend(const DecodeArgs& a, const WorkspaceLayout& L, const CUtensorMap& ta,
                            const CUtensorMap& tb, int max_records) {
    auto kern = attend_kernel<T, D, PAGED>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int sms = 0, smem_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    const int ctas_wanted = std::max(1, env_int("PA_DECODE_CTAS_PER_SM", 4));
    int nstage = env_int("PA_DECODE_STAGES", 0);
    if (nstage <= 0) {
        const long budget = (long)smem_sm / ctas_wanted - 1024;
        nstage = (int)((budget - 1040) / (long)(Geo<D>::kSlotBytes + sizeof(StageMeta) + 16));
    }
    nstage = std::max(2, std::min(nstage, 16));
    const size_t smem = attend_smem_bytes<D>(nstage);
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(attend)");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kAttnThreads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (per_sm < 1) return fail(PA_ERR_CUDA, "attention kernel does not fit on an SM (smem %zu)", smem);
    const int grid = std::max(1, std::min(per_sm * sms, max_records));

    AttnParams p;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    p.rec = reinterpret_cast<const int4*>(ws + L.records);
    p.header = reinterpret_cast<int*>(ws + L.header);
    p.tables = a.tables;
    p.MB = a.MB;
    p.B = a.B;
    p.NB = a.NB;
    p.req_ids = a.req_ids;
    p.S_max = a.S_max;
    p.q = a.q;
    p.H_q = a.H_q;
    p.G = a.H_q / a.H_kv;
    p.out = a.out;
    p.out_dtype = a.out_dtype;
    p.part_m2 = L.P > 1 ? reinterpret_cast<float*>(ws + L.part_m2) : nullptr;
    p.part_l = L.P > 1 ? reinterpret_cast<float*>(ws + L.part_l) : nullptr;
    p.part_acc = L.P > 1 ? reinterpret_cast<float*>(ws + L.part_acc) : nullptr;
    p.P = L.P;
    p.PT = L.PT;
    p.ctx_lens = a.ctx_lens;
    p.N = a.N;
    p.H_kv = a.H_kv;
    p.max_ctx = a.max_ctx;
    p.cap = a.paged ? a.MB * a.B : a.S_max;
    p.N_max = a.N_max;
    p.scale_log2 = (float)((double)a.scale * 1.4426950408889634);  // log2(e)
    p.nstage = nstage;
    p.wait_ns = wait_limit_ns();
    p.err = a.dev_err;

    if (a.attend_events && a.attend_events[0]) {
        e = cudaEventRecord(static_cast<cudaEvent_t>(a.attend_events[0]), a.stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    }
    e = launch_kernel(kern, dim3(grid), dim3(kAttnThreads), smem, a.stream, ta, tb, p);
    count_launch();
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    if (a.attend_events && a.attend_events[1]) {
        e = cudaEventRecord(static_cast<cudaEvent_t>(a.attend_events[1]), a.stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    }
    return PA_OK;
}

template <typename T, int D>
static pa_status dispatch_paged(const DecodeArgs& a, const WorkspaceLayout& L, const CUtensorMap& ta,
                                const CUtensorMap& tb, int maxrec) {
    return a.paged ? run_attend<T, D, true>(a, L, ta, tb, maxrec) : run_attend<T, D, false>(a, L, ta, tb, maxrec);
}

pa_status launch_decode(const DecodeArgs& a) {
    WorkspaceLayout L;
    if (!workspace_layout(a.N, a.H_q, a.H_kv, a.D, a.max_ctx, a.partition_tokens, &L))
        return fail(PA_ERR_INVALID, "invalid workspace arguments");
    if (a.ws_bytes < L.total) return fail(PA_ERR_INVALID, "workspace too small: %zu < %zu", a.ws_bytes, L.total);
    const int DH = a.D / 64;
    CUtensorMap ta, tb;
    std::memset(&ta, 0, sizeof ta);
    std::memset(&tb, 0, sizeof tb);
    const cuuint64_t esz = 2;
    if (a.paged) {
        // dims (innermost first): 64 columns, token (NB*B), column half, kv head, K/V
        cuuint64_t dims[5] = {64, (cuuint64_t)a.NB * a.B, (cuuint64_t)DH, (cuuint64_t)a.H_kv, 2};
        cuuint64_t str[4] = {(cuuint64_t)2 * a.H_kv * a.D * esz, 128, (cuuint64_t)a.D * esz,
                             (cuuint64_t)a.H_kv * a.D * esz};
        cuuint32_t box[5] = {64, (cuuint32_t)a.B, (cuuint32_t)DH, 1, 2};
        pa_status st = encode(&ta, a.kv_dtype, 5, a.pool, dims, str, box);
        if (st != PA_OK) return st;
        tb = ta;
    } else {
        cuuint64_t dims[4] = {64, (cuuint64_t)a.N_max * a.S_max, (cuuint64_t)DH, (cuuint64_t)a.H_kv};
        cuuint64_t str[3] = {(cuuint64_t)a.H_kv * a.D * esz, 128, (cuuint64_t)a.D * esz};
        cuuint32_t box[4] = {64, (cuuint32_t)kStageTok, (cuuint32_t)DH, 1};
        pa_status st = encode(&ta, a.kv_dtype, 4, a.k_buf, dims, str, box);
        if (st != PA_OK) return st;
        st = encode(&tb, a.kv_dtype, 4, a.v_buf, dims, str, box);
        if (st != PA_OK) return st;
    }

    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    int* header = reinterpret_cast<int*>(ws + L.header);
    int* nparts = reinterpret_cast<int*>(ws + L.nparts);
    int4* rec = reinterpret_cast<int4*>(ws + L.records);
    const int cap = a.paged ? a.MB * a.B : a.S_max;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // kPlanSlice sequences per CTA, at most one CTA per SM (larger slices beyond that)
    const int plan_ctas = std::min((a.N + kPlanSlice - 1) / kPlanSlice, std::max(sms, 1));
    cudaError_t e = launch_kernel(plan_kernel, dim3(plan_ctas), dim3(kPlanThreads), 0, a.stream, a.ctx_lens,
                                  a.paged ? nullptr : a.req_ids, a.N, a.H_kv, L.PT, a.max_ctx, cap, a.N_max,
                                  plan_bins(L.PT, a.max_ctx), header, rec, nparts, a.dev_err);
    count_launch();
    if (e != cudaSuccess) return cuda_fail(e, "plan launch");

    const long maxrec_l = (long)a.N * L.P * a.H_kv;
    const int maxrec = (int)std::min<long>(maxrec_l, 1L << 30);
    pa_status st;
    if (a.kv_dtype == PA_BF16)
        st = a.D == 128 ? dispatch_paged<__nv_bfloat16, 128>(a, L, ta, tb, maxrec)
                        : dispatch_paged<__nv_bfloat16, 64>(a, L, ta, tb, maxrec);
    else
        st = a.D == 128 ? dispatch_paged<__half, 128>(a, L, ta, tb, maxrec)
                        : dispatch_paged<__half, 64>(a, L, ta, tb, maxrec);
    if (st != PA_OK || L.P == 1) return st;
    return launch_partition_reduce(a.out, a.out_dtype, reinterpret_cast<float*>(ws + L.part_m2),
                                   reinterpret_cast<float*>(ws + L.part_l), reinterpret_cast<float*>(ws + L.part_acc),
                                   nparts, a.H_q, a.N * a.H_q, L.P, a.D, true, a.dev_err, a.stream);
}

}  // namespace pa

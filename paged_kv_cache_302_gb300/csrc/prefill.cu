// prefill.cu -- causal paged prefill attention on the sm_103a tensor cores (tcgen05 + TMEM).
//
// Method: PagedAttention explainer (0h-n0.github.io, arXiv 2309.06180), 実装のポイント:
// the paged kernel serves the prefill phase as well as decode -- a chunk of a
// sequence's newest tokens attends, causally, to the whole context through
// the block table.  Each query row follows the decode equation with its
// context cut at its own position.
//
// A query tile is 128 rows: 128/G query tokens times the G query heads of one
// KV head, so every K/V byte loaded serves G heads.  A CTA owns two consecutive
// query tiles, which share every K/V tile it loads (320 threads):
//   * warp 8 (TMA): both Q tiles once, then K and V of each 128-key tile into a
//     two-stage ring, through the block table, 128-byte swizzled; lane b issues
//     the copies of the tile's b-th KV block (V of a staged bf16 cache: two
//     boxes per tile from the staging area);
//   * warp 9 (MMA, one thread): S_w = Q_w K^T as tcgen05.mma (M 128, N 128,
//     K 16 steps) into TMEM columns [128w, 128w + 128), and O_w += P V with P
//     read from those same TMEM columns (the A operand) and V an MN-major
//     shared-memory operand; O_w sits in TMEM columns 256 + D w;
//   * warps 0-3 and 4-7 (softmax, one warpgroup per query tile): every thread
//     owns one TMEM lane = one query row; it reads its S row with tcgen05.ld,
//     masks causally, keeps the running maximum (rescaling O only when the
//     maximum grows by more than 2^8), and writes the probabilities back over S
//     (tcgen05.st).
// The value product is one fp16 product per 16 keys (P in fp16) when V is fp16:
// an fp16 cache, or a bf16 cache whose V stage_v_kernel has staged as fp16 in
// the caller's workspace.  Otherwise (a bf16 cache without a workspace, or a
// row whose values fp16 cannot hold exactly) P is a high and a low bf16 part
// and the product is P_hi V + P_lo V.
// Hand-offs are mbarriers; every wait is bounded.  Finally every thread reads
// its O row, divides by its exponential sum and stores the row.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "pa_device.cuh"

namespace pa {

constexpr int kPfRows = 128;     // query rows per query tile (tcgen05 M); a CTA owns two query tiles
constexpr int kPfKeys = 128;     // keys per tile (tcgen05 N of S, K of P V)
constexpr int kPfSoftmaxThreads = 256;  // two warpgroups, one per query tile: one thread per row / TMEM lane
constexpr int kPfThreads = kPfSoftmaxThreads + 64;  // + warp 8: TMA, warp 9: MMA
constexpr int kPfStages = 2;     // K and V stages in shared memory
constexpr uint32_t kTmemCols = 512;  // S/P of query tiles 0, 1 (128 columns each), then O_0, O_1 (D columns each)
constexpr uint32_t kRegion = kPfRows * 128;  // one [128 rows][64 columns] 16-bit swizzled region: 16 KB
constexpr int kGroupKeys = 32;               // keys per CTA of the V staging kernel (and per range-checked group)
constexpr int kWKeys = 256;                  // keys per tile of prefill_wide_kernel (tcgen05 N of its S)
constexpr int kStagePad = kWKeys;            // staged rows are written (zeros past the context) to a multiple of this

struct PrefillParams {
    const int32_t* tables;
    const int32_t* ctx_lens;
    const int32_t* q_start;
    int N, T, H_q, H_kv, G, TQ, B, MB, NB;
    void* out;
    int out_dtype;
    float scale_log2;
    uint64_t wait_ns;  // limit of the hand-off waits (the exit path waits with kWaitLimitNs)
    // bf16 V staged as fp16 by stage_v_kernel (null: V read from the pool, P split into two bf16 parts)
    const void* vstage;
    const int* vsplit;  // per (sequence, KV head): non-zero when its V could not be staged exactly
    int S_pad;          // keys per staged (sequence, KV head) row: a multiple of kStagePad
    int only_split;     // prefill_kernel: serve only the rows marked in vsplit (prefill_wide_kernel takes the rest)
    int max_q_len;      // longest chunk: prefill_wide_kernel's units per (sequence, KV head)
    int* err;
};

// ----------------------------------------------------------------------------- tcgen05 wrappers

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 encoding: address, leading and stride byte
// offsets in 16-byte units, descriptor version 1 at bit 46, layout code 2 at bit 61).
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16 with an fp32 accumulator.
__host__ __device__ constexpr uint32_t umma_idesc(bool bf16, int M, int N, bool b_mn_major) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Same, with the A operand (M rows x 16 k, two 16-bit elements per 32-bit column) read from TMEM.
__device__ __forceinline__ void umma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
        "r"(tmem_a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}

// Arrives on the mbarrier at this offset in every CTA of the cluster named by `mask` once the products issued so
// far have completed.
__device__ __forceinline__ void umma_commit_mc(uint32_t mbar, uint16_t mask) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                     "r"(mbar),
                 "h"(mask)
                 : "memory");
}

// 5-D tiled load multicast to the same shared-memory offset of every CTA of the cluster in `mask`; each destination
// CTA's mbarrier at offset `bar` counts the bytes it receives.
__device__ __forceinline__ void tma_load_5d_mc(uint32_t dst, const void* tmap, uint32_t bar, int c0, int c1, int c2,
                                               int c3, int c4, uint16_t mask, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8, %9;" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar), "h"(mask), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of both CTAs of the cluster: writes before it are visible to the other CTA after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ----------------------------------------------------------------------------- packed fp32 pairs

// d = a * b + c on two fp32 lanes at once (PTX fma.rn.f32x2).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Lane-wise unsigned maximum of two 16-bit pairs (PTX max.u16x2).
__device__ __forceinline__ uint32_t vmax_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// A pair of bfloat16 values as a pair of IEEE binary16 values, round to nearest even (exact when each value is
// zero or of magnitude in [2^-14, 65504]: a bfloat16 significand has 8 bits, a binary16 one 11).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xffff0000u);
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ----------------------------------------------------------------------------- V staging (bf16 caches)

// The value product takes P in fp16 (11-bit significand) when V is fp16.  A bf16 cache's V is staged as fp16 by
// this kernel, per (sequence, KV head) in key order: stage[s * H_kv + h][t][D], t < S_pad, zeros past the context.
// bf16 -> fp16 is exact for zero and for magnitudes in [2^-14, 65504].  A (sequence, KV head) row with a magnitude
// of 65536 or more (fp16 would overflow; also inf and NaN), or with a 32-key group of context keys whose
// magnitudes are all below 2^-10 (fp16 subnormals would drop bits), is marked in `split` (zeroed before this
// kernel): the prefill kernel's CTAs of that row then read V from the pool and take P as a high and a low bf16
// part (two products), as every CTA does when nothing is staged.
// One CTA per 32 keys of a sequence and group of up to 8 KV heads.  One TMA box per KV block brings the block's V
// rows of those heads into shared memory ([head][column half][token][64 columns], unswizzled; heads past H_kv
// read as zeros), then the 256 threads convert 16-byte chunks and write whole 256-byte rows of the staging area.
// (Plain loads through the block table, a warp per head, moved ~2.5 TB/s; the attention kernel's TMA boxes over
// the same per-head rows move ~6.8 TB/s.)
constexpr int kStageThreads = 256;
constexpr int kStageHeads = 8;  // KV heads per CTA, one TMA box per KV block

template <int D>
__global__ void __launch_bounds__(kStageThreads) stage_v_kernel(const __grid_constant__ CUtensorMap tm_v,
                                                                const int32_t* __restrict__ tables,
                                                                const int32_t* __restrict__ ctx_lens, int H_kv,
                                                                int B, int MB, int NB, int S_pad,
                                                                uint16_t* __restrict__ stage,
                                                                int* __restrict__ split, uint64_t wait_ns, int* err) {
    constexpr int DH = D / 64;
    constexpr int kRowChunks = DH * 8;  // 16-byte chunks per V row
    extern __shared__ __align__(128) uint8_t vbuf[];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t hmax[kStageHeads];
    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x;
    const int s = blockIdx.z, h0 = blockIdx.y * kStageHeads, t0 = blockIdx.x * kGroupKeys;
    const int hb = min(kStageHeads, H_kv), nh = min(hb, H_kv - h0);
    int ctx = ctx_lens[s];
    if (ctx < 0 || ctx > MB * B) ctx = 0;  // flagged by the prefill kernel, which then computes nothing
    if (t0 >= (ctx + kStagePad - 1) / kStagePad * kStagePad) return;  // uniform per CTA: past the last tile read
    const int nvalid = max(0, min(kGroupKeys, ctx - t0));
    const int nblk = (nvalid + B - 1) / B;  // KV blocks holding this CTA's context keys
    const uint32_t box_bytes = 128u * B * DH * hb;
    const uint32_t bar_s = smem_addr(&bar), buf_s = smem_addr(vbuf);
    if (tid < kStageHeads) hmax[tid] = 0;
    if (tid == 0) {
        mbar_init(bar_s, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        mbar_arrive_expect_tx(bar_s, nblk * box_bytes);
        const uint64_t pol = policy_evict_first();
        for (int b = 0; b < nblk; ++b) {
            int e = tables[(size_t)s * MB + t0 / B + b];
            if ((unsigned)e >= (unsigned)NB) {
                flag_error(err, PA_DEV_ERR_BLOCK);
                e = NB;  // past the tensor: TMA fills zeros
            }
            tma_load_5d(buf_s + b * box_bytes, &tm_v, bar_s, 0, e * B, 0, h0, 1, pol);
        }
    }
    if (!mbar_wait_bounded(bar_s, 0, nullptr, wait_ns)) {
        if (tid == 0) flag_error(err, PA_DEV_ERR_TIMEOUT);
        mbar_wait_bounded(bar_s, 0, nullptr);  // the copies land in this CTA's shared memory: let them
    }
    // chunk c: row (key tt = (c / kRowChunks) % 32, head hh = c / (kRowChunks * 32)), column chunk c % kRowChunks;
    // with 256 threads every pass over the chunks covers a single head
    constexpr int kPerHead = kRowChunks * kGroupKeys;
    for (int c = tid; c < hb * kPerHead; c += kStageThreads) {
        const int hh = c / kPerHead, tt = (c / kRowChunks) % kGroupKeys, q = c % kRowChunks;
        const int half = q / 8, cq = q % 8;
        uint4 x = make_uint4(0, 0, 0, 0);
        if (tt < nvalid)
            x = *reinterpret_cast<const uint4*>(vbuf + (tt / B) * box_bytes +
                                                (((hh * DH + half) * B + tt % B) * 128 + cq * 16));
        uint32_t m = vmax_u16x2(vmax_u16x2(x.x & 0x7fff7fffu, x.y & 0x7fff7fffu),
                                vmax_u16x2(x.z & 0x7fff7fffu, x.w & 0x7fff7fffu));
        m = __reduce_max_sync(0xffffffffu, max(m & 0xffffu, m >> 16));
        if ((tid & 31) == 0) atomicMax(&hmax[hh], m);
        if (hh < nh)
            reinterpret_cast<uint4*>(stage + ((size_t)(s * H_kv + h0 + hh) * S_pad + t0 + tt) * D)[q] =
                make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z), bf16x2_to_f16x2(x.w));
    }
    __syncthreads();
    // 0x4780: bf16 magnitude bits of 65536; 0x3a80: of 2^-10
    if (tid < nh && nvalid > 0 && (hmax[tid] >= 0x4780u || hmax[tid] < 0x3a80u))
        atomicOr(split + s * H_kv + h0 + tid, 1);
}

// ----------------------------------------------------------------------------- kernel

template <typename T, int D>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                                const __grid_constant__ CUtensorMap tm_kv,
                                                                const __grid_constant__ CUtensorMap tm_kv_blk,
                                                                const __grid_constant__ CUtensorMap tm_vs,
                                                                const PrefillParams p) {
    constexpr int DH = D / 64;          // 64-column halves of a head row
    constexpr int NK = D / 16;          // k-steps of S = Q K^T
    constexpr int NT = kPfKeys / 16;    // k-steps of O += P V
    constexpr int NS = kPfStages;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    // The value product takes P in fp16 (11-bit significand, relative L2 error ~1.4e-4) when V is fp16: an fp16
    // cache, or a bf16 cache whose V stage_v_kernel staged as fp16.  A CTA of a bf16 cache with nothing staged, or
    // of a (sequence, KV head) row the staging kernel marked, reads V from the pool and takes P as a high and a low
    // bf16 part, two products (a single bf16 P, 8 bits, would put the error near 1e-3).  The choice is made once per
    // CTA, outside the loops: a choice per key tile inside them measured ~7 % slower (the issuing thread lost its
    // straight-line code), one per 32 keys a quarter slower.
    constexpr uint32_t idesc_s = umma_idesc(kBf16, kPfRows, kPfKeys, false);
    constexpr uint32_t idesc_o16 = umma_idesc(false, kPfRows, D, true);
    constexpr uint32_t idesc_obf = umma_idesc(true, kPfRows, D, true);
    constexpr uint32_t kTile = DH * kRegion;  // one Q tile (128 rows x D), or one K or V tile (128 keys x D)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_addr(base);
    // Q[2] | K[NS] | V[NS] | barriers
    const uint32_t sQ0 = sb, sK0 = sQ0 + 2 * kTile, sV0 = sK0 + NS * kTile, sBar = sV0 + NS * kTile;
    // barriers: q; k_full, v_full, k_free, v_free [NS]; s_full, pv_done, p_ready [2] (one per query tile);
    // mma_done (the MMA thread's last commit: every product it issued has completed)
    const uint32_t qbar = sBar, kfull0 = qbar + 8, vfull0 = kfull0 + 8 * NS, kfree0 = vfull0 + 8 * NS,
                   vfree0 = kfree0 + 8 * NS, sfull0 = vfree0 + 8 * NS, pvd0 = sfull0 + 16, prd0 = pvd0 + 16,
                   mmadone = prd0 + 16;
    constexpr int kBars = 1 + 4 * NS + 6 + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + (sBar - sb) + 8 * kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + (sBar - sb) + 8 * kBars + 4);
    // K and V tiles whose copies the TMA warp has issued (tile t uses stage t % NS), kept in shared memory for
    // the exit path rather than in registers
    volatile int* armed = abort_flag + 1;

    griddep_wait();
    griddep_launch_dependents();
    // the marks are written by the staging kernel launched just before: read them only after the wait above
    const bool staged = kBf16 && p.vstage != nullptr;
    const bool split = kBf16 && (!staged || p.vsplit[blockIdx.z * p.H_kv + blockIdx.y] != 0);
    const bool vstaged = staged && !split;  // V tiles come from the staging area
    if (p.only_split && !split) return;     // uniform per CTA, before any allocation
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.z, g = blockIdx.y;
    const int qs = p.q_start[s], q_len = p.q_start[s + 1] - qs;
    // query-tile pairs are dispatched latest first: under the causal mask they have the most keys, so the last
    // CTAs to run are the shortest
    const int tok0 = (gridDim.x - 1 - blockIdx.x) * 2 * p.TQ;  // first query token of tile 0; tile 1 at tok0 + TQ
    if (tok0 >= q_len) return;  // uniform per CTA, before any allocation
    const int ctx = p.ctx_lens[s];
    if (q_len > ctx || ctx > p.MB * p.B || q_len < 0) {
        if (tid == 0) flag_error(p.err, PA_DEV_ERR_CTX);
        return;
    }
    const int pos0 = ctx - q_len + tok0;                         // position of the CTA's first query token
    const int last_tok = min(tok0 + 2 * p.TQ, q_len) - 1;
    const int nkeys = ctx - q_len + last_tok + 1;                // keys the CTA's last query sees
    const int ntiles = (nkeys + kPfKeys - 1) / kPfKeys;
    auto st = [](int j) { return (uint32_t)(j % NS); };
    auto ph = [](int j) { return (uint32_t)((j / NS) & 1); };
    // With B = 8 the K and V tiles are stored block by block, [block][half][8 rows][128 bytes], and one copy
    // brings a whole block; otherwise each tile holds one 128-key region per 64-column half, [half][128 rows][128 B]
    // (one copy per block and half), which measured faster for the value product at B = 16 and 32.  A staged V
    // tile always has the second layout.
    const bool k_blk = p.B == 8, v_blk = p.B == 8 && !vstaged;
    const uint32_t blk_bytes = (uint32_t)DH * p.B * 128;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int i = 0; i < kBars; ++i) mbar_init(sBar + 8 * i, 1);
        mbar_init(prd0, kPfRows);
        mbar_init(prd0 + 8, kPfRows);
        *abort_flag = 0;
        armed[0] = armed[1] = 0;
        fence_mbar_init();
    }
    // rows past TQ*G (when G does not divide 128) are never loaded: clear them once in both query tiles
    if (warp < 8)
        for (int r = p.TQ * p.G + (warp & 3); r < kPfRows; r += 4)
            for (int dh = 0; dh < DH; ++dh)
                if (lane < 8)
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sQ0 + (warp >> 2) * kTile +
                                                                                  dh * kRegion + r * 128 + lane * 16),
                                 "r"(0)
                                 : "memory");
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;  // columns: S/P of query tile w at 128 w, O_w at 256 + D w
    auto waited = [&](uint32_t bar, uint32_t parity) {
        const bool w = mbar_wait_bounded(bar, parity, abort_flag, p.wait_ns);
        if (!w) *abort_flag = 1;
        return w;
    };
    bool ok = true;

    if (warp == 8) {
        // ------------------------------------------------------------ TMA producer
        const uint64_t pol = policy_evict_first();
        if (lane == 0) {
            mbar_arrive_expect_tx(qbar, (uint32_t)2 * DH * p.G * p.TQ * 128);
            for (int w = 0; w < 2; ++w)
                for (int dh = 0; dh < DH; ++dh)
                    tma_load_4d(sQ0 + w * kTile + dh * kRegion, &tm_q, qbar, 0, dh, g * p.G, qs + tok0 + w * p.TQ,
                                policy_evict_normal());
        }
        // Lane b issues the copies of the tile's b-th KV block.
        auto table_entry = [&](int t) {
            const int k0 = t * kPfKeys;
            const int nblk = min(kPfKeys, ctx - k0 + p.B - 1) / p.B;  // blocks holding keys of this tile
            int e = lane < nblk ? p.tables[(size_t)s * p.MB + k0 / p.B + lane] : 0;
            if (lane < nblk && (unsigned)e >= (unsigned)p.NB) {
                flag_error(p.err, PA_DEV_ERR_BLOCK);
                e = p.NB;  // past the tensor: TMA fills zeros
            }
            return e;
        };
        int mine = table_entry(0);
        for (int t = 0; t < ntiles && ok; ++t) {
            const int nblk = min(kPfKeys, ctx - t * kPfKeys + p.B - 1) / p.B;
            const int cur = mine;
            if (t + 1 < ntiles) mine = table_entry(t + 1);  // in flight while this tile's copies are issued
            const uint32_t bytes = (uint32_t)nblk * DH * p.B * 128;
            const uint32_t b = st(t);
            for (int which = 0; which < 2 && ok; ++which) {
                // stage t % NS is free once both query tiles' S_{t-NS} (for K) / PV_{t-NS} (for V) are done
                if (t >= NS) ok = waited((which ? vfree0 : kfree0) + 8 * b, ph(t - NS));
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const uint32_t bar = (which ? vfull0 : kfull0) + 8 * b;
                const uint32_t dst = (which ? sV0 : sK0) + b * kTile;
                if (which && vstaged) {
                    // the staged V tile: 128 keys of this (sequence, KV head), one copy per 64-column half
                    if (lane == 0) {
                        armed[1] = t + 1;
                        mbar_arrive_expect_tx(bar, kTile);
                        for (int dh = 0; dh < DH; ++dh)
                            tma_load_4d(dst + dh * kRegion, &tm_vs, bar, 0, dh, t * kPfKeys, s * p.H_kv + g, pol);
                    }
                    __syncwarp();
                    continue;
                }
                if (lane == 0) {
                    armed[which] = t + 1;  // expect_tx and every copy below, with no wait in between
                    mbar_arrive_expect_tx(bar, bytes);
                }
                __syncwarp();
                if (lane < nblk) {
                    if (which ? v_blk : k_blk)
                        tma_load_5d(dst + (uint32_t)lane * blk_bytes, &tm_kv_blk, bar, 0, cur * p.B, 0, g, which, pol);
                    else
                        for (int dh = 0; dh < DH; ++dh)
                            tma_load_5d(dst + dh * kRegion + (uint32_t)lane * p.B * 128, &tm_kv, bar, 0, cur * p.B, dh,
                                        g, which, pol);
                }
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        // S_w(j) = Q_w K_j^T goes to TMEM buffer w and is overwritten there by P_w(j); O_w += P_w(j) V_j.
        // S_w(j+1) reuses the buffer once PV_w(j) has read P_w(j).
        // Descriptors are built once per operand and advanced per k-step by adding the byte offset / 16 to their
        // 14-bit address field (shared-memory addresses stay below 256 KB, so the field never carries); building
        // both 64-bit descriptors per instruction slowed the single issuing thread (measured 789 -> 824 TFLOP/s).
        const uint64_t dq0 = umma_desc(sQ0, 16, 1024), dq1 = umma_desc(sQ0 + kTile, 16, 1024);
        auto issue_s = [&](int w, int j) {
            const uint32_t kb = sK0 + st(j) * kTile;
            const uint64_t dq = w ? dq1 : dq0;
            const uint64_t dk = k_blk ? umma_desc(kb, 16, blk_bytes) : umma_desc(kb, 16, 1024);
#pragma unroll
            for (int ks = 0; ks < NK; ++ks) {
                constexpr uint32_t kR16 = kRegion >> 4;
                const uint32_t qoff = (ks >> 2) * kR16 + (ks & 3) * 2;
                const uint32_t koff = k_blk ? (ks >> 2) * 64 + (ks & 3) * 2 : qoff;
                umma_f16(tmem + (uint32_t)w * kPfKeys, dq + qoff, dk + koff, idesc_s, ks > 0);
            }
            umma_commit(sfull0 + 8 * w);
            if (w == 1) umma_commit(kfree0 + 8 * st(j));  // K_j has served both query tiles
        };
        // O_w += P V with P read from TMEM: one fp16 product per 16 keys, or (split) P_hi V + P_lo V in bf16
        auto issue_pv = [&](int w, int j, auto split_c) {
            const uint32_t vb = sV0 + st(j) * kTile;
            const uint32_t pcol = tmem + (uint32_t)w * kPfKeys;
            const uint32_t ocol = tmem + 2 * kPfKeys + (uint32_t)w * D;
            const uint64_t dv = !v_blk ? umma_desc(vb, kRegion, 1024) : umma_desc(vb, 1024, blk_bytes);
            const uint32_t vstep = !v_blk ? (16 * 128) >> 4 : (2 * blk_bytes) >> 4;
            constexpr bool kSplit = decltype(split_c)::value;
#pragma unroll
            for (int ks = 0; ks < NT; ++ks) {
                const uint64_t vdesc = dv + (uint64_t)(ks * vstep);
                umma_f16_ta(ocol, pcol + ks * 8, vdesc, kSplit ? idesc_obf : idesc_o16, (j > 0 || ks > 0));
                if (kSplit) umma_f16_ta(ocol, pcol + kPfKeys / 2 + ks * 8, vdesc, idesc_obf, 1u);
            }
            umma_commit(pvd0 + 8 * w);
            if (w == 1) umma_commit(vfree0 + 8 * st(j));
        };
        if (lane == 0) {
            ok = waited(qbar, 0) && waited(kfull0, 0);
            tc_fence_after();
            if (ok) {
                issue_s(0, 0);
                issue_s(1, 0);
            }
            // the tile loop, one copy per kind of value product
            auto tiles = [&](auto split_c) {
                for (int j = 0; j < ntiles && ok; ++j) {
                    const bool more = j + 1 < ntiles;
                    for (int w = 0; w < 2 && ok; ++w) {
                        ok = waited(prd0 + 8 * w, (uint32_t)(j & 1)) &&
                             (w == 1 || waited(vfull0 + 8 * st(j), ph(j)));
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(w, j, split_c);
                        if (more) {
                            ok = (w == 1 || waited(kfull0 + 8 * st(j + 1), ph(j + 1))) &&
                                 waited(pvd0 + 8 * w, (uint32_t)(j & 1));
                            tc_fence_after();
                            if (ok) issue_s(w, j + 1);
                        }
                    }
                }
            };
            if (split)
                tiles(std::true_type{});
            else
                tiles(std::false_type{});
            // arrives once every product issued above has completed (at once when none was issued)
            umma_commit(mmadone);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax: warpgroup w owns query tile w
        // thread = query row = TMEM lane
        const int wg = warp >> 2;
        const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t t_s = t_lane + (uint32_t)wg * kPfKeys;
        const uint32_t t_o = t_lane + 2 * kPfKeys + (uint32_t)wg * D;
        const int r = tid & (kPfRows - 1);
        const int qtok = wg * p.TQ + r / p.G;  // query token within the CTA
        const bool row_ok = r < p.TQ * p.G && tok0 + qtok < q_len;
        const int qpos = row_ok ? pos0 + qtok : -1;  // -1 masks every key
        const int first_pos = pos0 + wg * p.TQ;     // position of the tile's first token
        const float NEG_INF = -INFINITY;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        float m_ref = NEG_INF, l = 0.f;
        // the tile loop, one copy per kind of value product (the choice is made once, outside it)
        auto tiles = [&](auto split_c) {
            for (int j = 0; j < ntiles; ++j) {
                const int k0 = j * kPfKeys;
                ok = waited(sfull0 + 8 * wg, (uint32_t)(j & 1)) && ok;
                tc_fence_after();
                float v[kPfKeys];
                {
                    uint32_t* u = reinterpret_cast<uint32_t*>(v);
#pragma unroll
                    for (int c = 0; c < kPfKeys / 32; ++c)
                        asm volatile(
                            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
                            "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
                            "%28, %29, %30, %31}, [%32];"
                            : "=r"(u[32 * c + 0]), "=r"(u[32 * c + 1]), "=r"(u[32 * c + 2]), "=r"(u[32 * c + 3]),
                              "=r"(u[32 * c + 4]), "=r"(u[32 * c + 5]), "=r"(u[32 * c + 6]), "=r"(u[32 * c + 7]),
                              "=r"(u[32 * c + 8]), "=r"(u[32 * c + 9]), "=r"(u[32 * c + 10]), "=r"(u[32 * c + 11]),
                              "=r"(u[32 * c + 12]), "=r"(u[32 * c + 13]), "=r"(u[32 * c + 14]), "=r"(u[32 * c + 15]),
                              "=r"(u[32 * c + 16]), "=r"(u[32 * c + 17]), "=r"(u[32 * c + 18]), "=r"(u[32 * c + 19]),
                              "=r"(u[32 * c + 20]), "=r"(u[32 * c + 21]), "=r"(u[32 * c + 22]), "=r"(u[32 * c + 23]),
                              "=r"(u[32 * c + 24]), "=r"(u[32 * c + 25]), "=r"(u[32 * c + 26]), "=r"(u[32 * c + 27]),
                              "=r"(u[32 * c + 28]), "=r"(u[32 * c + 29]), "=r"(u[32 * c + 30]), "=r"(u[32 * c + 31])
                            : "r"(t_s + c * 32)
                            : "memory");
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                }
                // only tiles that reach past the tile's first position need the causal mask
                const bool masked = k0 + kPfKeys - 1 > first_pos || !row_ok;
                if (masked) {
#pragma unroll
                    for (int i = 0; i < kPfKeys; ++i) v[i] = k0 + i <= qpos ? v[i] : NEG_INF;
                }
                float mx[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
                for (int i = 0; i < kPfKeys; i += 8) {
                    mx[0] = fmax3(mx[0], v[i], v[i + 1]);
                    mx[1] = fmax3(mx[1], v[i + 2], v[i + 3]);
                    mx[2] = fmax3(mx[2], v[i + 4], v[i + 5]);
                    mx[3] = fmax3(mx[3], v[i + 6], v[i + 7]);
                }
                const float m_tile = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * p.scale_log2;
                float m_new = m_ref;
                if (j == 0 || m_tile > m_ref + 8.f) m_new = fmaxf(m_ref, m_tile);
                const float alpha = (j == 0 || m_new == m_ref) ? 1.f : fast_exp2(m_ref - m_new);
                m_ref = m_new;
                const float m_use = m_new == NEG_INF ? 0.f : m_new;
                const float2 nm2 = make_float2(-m_use, -m_use);
                // P overwrites S in TMEM: fp16 in the buffer's first 64 columns; split, the high bf16 parts there and
                // the low parts in the next 64
                float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                auto write_p = [&](auto split_c) {
                    constexpr bool kSplit = decltype(split_c)::value;
                    using PT = typename std::conditional<kSplit, __nv_bfloat16, __half>::type;
#pragma unroll
                    for (int c = 0; c < kPfKeys / 32; ++c) {
                        uint32_t hi[16], lo[16];
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float2 x = ffma2(make_float2(v[32 * c + i], v[32 * c + i + 1]), sc2, nm2);
                            x.x = fast_exp2(x.x);
                            x.y = fast_exp2(x.y);
                            ls[(i >> 1) & 1] = fadd2(ls[(i >> 1) & 1], x);
                            hi[i / 2] = Mma<PT>::pack(x.x, x.y);
                            if (kSplit) {
                                const float2 f = fsub2(x, Mma<PT>::unpack(hi[i / 2]));
                                lo[i / 2] = Mma<PT>::pack(f.x, f.y);
                            }
                        }
                        tmem_st16(t_s + c * 16, hi);
                        if (kSplit) tmem_st16(t_s + kPfKeys / 2 + c * 16, lo);
                    }
                };
                write_p(split_c);
                const float2 lsum = fadd2(ls[0], ls[1]);
                l = fmaf(l, alpha, lsum.x + lsum.y);
                // O_w is rescaled (rarely: only when the maximum grew by more than 2^8) once PV_w(j-1) has landed
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                    ok = waited(pvd0 + 8 * wg, (uint32_t)((j - 1) & 1)) && ok;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        float o[32];
                        tmem_ld32(t_o + c * 32, o);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tmem_st32(t_o + c * 32, o);
                    }
                }
                // V rows past the context may hold anything (even NaN): tile 0's warpgroup zeroes them before either
                // query tile's PV (PV_0 is issued first) can meet them with P = 0
                const int nvalid = min(kPfKeys, ctx - k0);
                if (wg == 0 && nvalid < kPfKeys && !vstaged) {  // a staged tile has zeros there already
                    ok = waited(vfull0 + 8 * st(j), ph(j)) && ok;
                    const uint32_t vb = sV0 + st(j) * kTile;
                    for (int rr = nvalid + (warp & 3); rr < kPfKeys; rr += 4)
                        for (int dh = 0; dh < DH; ++dh)
                            if (lane < 8)
                                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                                                 v_blk ? vb + (uint32_t)(rr / p.B) * blk_bytes +
                                                             (uint32_t)(dh * p.B + rr % p.B) * 128 + lane * 16
                                                       : vb + dh * kRegion + rr * 128 + lane * 16),
                                             "r"(0)
                                             : "memory");
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(prd0 + 8 * wg);
                if (*abort_flag) break;
            }
        };
        if (split)
            tiles(std::true_type{});
        else
            tiles(std::false_type{});
        const int jl = ntiles - 1;
        if (ok) ok = waited(pvd0 + 8 * wg, (uint32_t)(jl & 1));
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
            tc_fence_after();
            const float inv = 1.f / l;
            const size_t orow = ((size_t)(qs + tok0 + qtok) * p.H_q + (size_t)g * p.G + (r % p.G)) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tmem_ld32(t_o + c * 32, o);
                if (row_ok) {
                    if (p.out_dtype == PA_F32) {
                        // 256-bit stores: each lane writes whole 32-byte sectors of its row (the host checks
                        // that `out` is 32-byte aligned; rows are D floats long)
                        float* dst = static_cast<float*>(p.out) + orow + c * 32;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 8 * i),
                                         "f"(o[8 * i] * inv), "f"(o[8 * i + 1] * inv), "f"(o[8 * i + 2] * inv),
                                         "f"(o[8 * i + 3] * inv), "f"(o[8 * i + 4] * inv), "f"(o[8 * i + 5] * inv),
                                         "f"(o[8 * i + 6] * inv), "f"(o[8 * i + 7] * inv)
                                         : "memory");
                    } else {
                        T* dst = static_cast<T*>(p.out) + orow + c * 32;
#pragma unroll
                        for (int i = 0; i < 32; ++i) dst[i] = from_float<T>(o[i] * inv);
                    }
                }
            }
        }
    }
    // Nothing issued may still be running when TMEM and shared memory are released: the tensor-core products
    // (the MMA thread's last commit) and the copies (the last arm of every stage: stage b's arms are tiles
    // b, b + NS, ...; each was consumed before the next was armed, so only the last can be in flight).  After a
    // wait ran out these can be anywhere; in a call that ran to completion they have all landed.
    if (warp == 9 && lane == 0) mbar_wait_bounded(mmadone, 0, nullptr);
    if (warp == 8 && lane == 0) {
        mbar_wait_bounded(qbar, 0, nullptr);
        for (int which = 0; which < 2; ++which) {
            const int n = armed[which];
            for (int b = 0; b < NS && b < n; ++b)
                mbar_wait_bounded((which ? vfull0 : kfull0) + 8 * b, ph(b + (n - 1 - b) / NS * NS), nullptr);
        }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok && !*abort_flag);
    if (!ok && tid == 0) flag_error(p.err, PA_DEV_ERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ----------------------------------------------------------------------------- one query tile, 256-key tiles

// prefill_wide_kernel: the same computation for the rows whose value product takes P in fp16 (an fp16 cache, or a
// bf16 cache's rows that stage_v_kernel converted; the rows it marked are left to prefill_kernel).  A CTA works on
// one 128-row query tile of one (sequence, KV head) at a time.  S = Q K^T of 256 keys at once: a tcgen05.mma of
// N = 256 per 16 columns of the head dim runs the tensor core at its full rate, where N = 128 products chained into
// one accumulator (prefill_kernel's) ran at ~60 % of it.  S sits in TMEM columns [0, 256) and P (fp16) in columns of
// its own, [384, 512), so the S product of the next key tile is issued as soon as the softmax has read S into
// registers and runs while the exponentials are computed; O += P V (16 keys per product, O in columns
// [256, 256 + D)) follows once P is written.
// The kernel is persistent and runs as clusters of two CTAs, one CTA per SM: cluster c takes units c, c + clusters,
// ... (ordered as wide_unit states), a unit being two neighbouring query tiles, one per CTA.  Both CTAs need the same
// K and V tiles: each copies half of every tile's blocks into both CTAs' shared memory (TMA multicast), which halves
// the copies and the L2 reads per SM.  The set-up (TMEM, barriers) is paid once.  Between units the next query tile
// is loaded while the softmax works on the last key tile.  Barrier phases follow counters that run across units
// (units, key tiles, ring items).
//   * warps 0-7 (softmax): warp w owns TMEM lanes 32 (w % 4) .. + 31 (query rows) and key columns 128 (w / 4) ..
//     + 127 of each tile; the two warps of a row share their row maxima through shared memory when either grew, so
//     both halves of P have one scale, and at the end their exponential sums; each stores D / 2 columns of O;
//   * warp 8 (TMA): Q, then the K and V tiles into a ring of three 256-key slots in the order the products consume
//     them (per unit: K_0, then K_{j+1}, V_j, ..., then the last V).  A slot is laid out [8-row group][column half]
//     [8 rows][128 B], so one copy brings a whole KV block (both column halves of its B rows): lane b issues the
//     copy of the tile's b-th block when b has this CTA's parity; a staged V tile is two copies of 128 keys, one
//     per CTA.  A slot is free again once both CTAs' products have read it;
//   * warp 9 (MMA, one thread): per unit S_0, then S_{j+1} once the softmax has read S_j and PV_j once P_j is
//     written.
constexpr int kWSlots = 3;                   // ring slots, each one 256-key K or V tile
constexpr uint32_t kWRegion = kWKeys * 128;  // 256 rows of 64 16-bit columns: 32 KB per column half
constexpr uint32_t kWColO = 256;             // TMEM columns of O (D of them)
constexpr uint32_t kWColP = 384;             // TMEM columns of P: 256 keys of fp16, two per column
constexpr int kWBars = 14;                   // q, q_free, full/free per slot, s_full, s_free, p_ready, pv_done,
                                             // o_free, mma_done

// Ring item i of a unit, in the order the products consume the tiles: K_0, then K_{j+1} and V_j for j = 0 .. n-2,
// then V_{n-1}.
__device__ __forceinline__ void wide_item(int i, int n, int& which, int& tile) {
    if (i == 0) {
        which = 0;
        tile = 0;
    } else if (i == 2 * n - 1) {
        which = 1;
        tile = n - 1;
    } else {
        which = ((i - 1) & 1) ? 1 : 0;
        tile = ((i - 1) >> 1) + (which ? 0 : 1);
    }
}

// Named barrier `id` over the 64 threads of the two softmax warps that hold the same query rows (warps w and
// w + 4, ids 1-4); the second form also returns whether any of them passed `flag`.
__device__ __forceinline__ void pair_sync(uint32_t id) { asm volatile("bar.sync %0, 64;" ::"r"(id) : "memory"); }
__device__ __forceinline__ bool pair_sync_any(uint32_t id, bool flag) {
    uint32_t any;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %2, 0;\n\tbar.red.or.pred q, %1, 64, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(any)
        : "r"(id), "r"((uint32_t)flag)
        : "memory");
    return any != 0;
}

template <int D>
static constexpr size_t wide_smem_bytes() {
    // alignment slack, Q, ring, barriers, TMEM address / abort flag / armed counts, row exchange [2][128]
    return 1024 + (size_t)(D / 64) * kRegion + (size_t)kWSlots * (D / 64) * kWRegion + 8 * kWBars + 16 + 2 * 128 * 4;
}

// A unit of prefill_wide_kernel is a pair of neighbouring query tiles of one (sequence, KV head), one per CTA of a
// cluster: pair px (counted from the last) holds query tiles x = 2 px (rank 0, the later one: the most keys) and
// 2 px + 1 (rank 1).  Unit w has px = w % npx: the clusters running at one time work on neighbouring pairs of the
// same row and share its K and V in L2 (an order with the sequence fastest read K and V from DRAM once per query
// tile), and each cluster's units (w = c + clusters i) cycle through long and short query tiles alike.  Both CTAs
// load the pair's key tiles (as many as rank 0's rows need); rank 1's keys past its own causal range are masked.
// A CTA whose tile holds no row of the chunk (rank 0's past its end, or rank 1's at tok0 < 0 when the row has an
// odd number of query tiles) still takes its part in the copies and computes no row.
struct WideUnit {
    int s, g, qs, q_len, tok0, ctx, pos0, ntiles;
};
enum { kUnitOk = 0, kUnitEmpty = 1, kUnitBadCtx = 2, kUnitOther = 3 };

template <bool kBf16>
__device__ __forceinline__ int wide_unit(const PrefillParams& p, int nx, int npx, int w, int rank, WideUnit& u) {
    const int rest = w / npx;
    const int tok_pair = (nx - 1 - 2 * (w % npx)) * p.TQ;  // rank 0's first query token
    u.g = rest % p.H_kv;
    u.s = rest / p.H_kv;
    u.qs = p.q_start[u.s];
    u.q_len = p.q_start[u.s + 1] - u.qs;
    // empty when both tiles lie past the chunk (rank 1's, the earlier one, included); rank 0's tile alone may
    if (u.q_len <= 0 || tok_pair - p.TQ >= u.q_len) return kUnitEmpty;
    u.ctx = p.ctx_lens[u.s];
    if (u.q_len > u.ctx || u.ctx > p.MB * p.B || u.q_len < 0) return kUnitBadCtx;
    // a bf16 row that was not staged (or that the staging marked) is prefill_kernel's, with the split P
    if (kBf16 && (p.vstage == nullptr || p.vsplit[u.s * p.H_kv + u.g] != 0)) return kUnitOther;
    u.tok0 = tok_pair - rank * p.TQ;                                  // this CTA's query tile
    u.pos0 = u.ctx - u.q_len + u.tok0;                                // position of its first query token
    const int nkeys = u.ctx - u.q_len + min(tok_pair + p.TQ, u.q_len);  // keys the pair's last query sees
    u.ntiles = (nkeys + kWKeys - 1) / kWKeys;
    return kUnitOk;
}

template <typename T, int D>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPfThreads, 1)
    prefill_wide_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kvg,
                        const __grid_constant__ CUtensorMap tm_vsg, const PrefillParams p) {
    constexpr int DH = D / 64;        // 64-column halves of a head row
    constexpr int NK = D / 16;        // k-steps of S = Q K^T
    constexpr int NT = kWKeys / 16;   // k-steps of O += P V
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t idesc_s = umma_idesc(kBf16, kPfRows, kWKeys, false);
    constexpr uint32_t idesc_o = umma_idesc(false, kPfRows, D, true);
    constexpr uint32_t kQ = DH * kRegion;      // the query tile: 128 rows x D
    constexpr uint32_t kSlot = DH * kWRegion;  // a ring slot: 256 keys x D, [8-row group][half][8 rows][128 B]
    constexpr uint32_t kGroup = DH * 1024;     // bytes per 8-row group of a slot
    static_assert(wide_smem_bytes<D>() <= 232448, "shared memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_addr(base);
    // Q | ring[kWSlots] | barriers
    const uint32_t sQ = sb, sR = sQ + kQ, sBar = sR + kWSlots * kSlot;
    const uint32_t qbar = sBar, qfree = qbar + 8, full0 = qfree + 8, free0 = full0 + 8 * kWSlots,
                   sfull = free0 + 8 * kWSlots, sfree = sfull + 8, prdy = sfree + 8, pvd = prdy + 8, ofree = pvd + 8,
                   mmadone = ofree + 8;
    uint8_t* extra = base + (sBar - sb) + 8 * kWBars;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(extra);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(extra + 4);
    volatile int* armed = abort_flag + 1;    // ring items whose copies the TMA warp has issued, for the exit path
    volatile int* armed_q = abort_flag + 2;  // query tiles the TMA warp has loaded, likewise
    float* xrow = reinterpret_cast<float*>(extra + 16);  // [half][row]: row maxima, at the end exponential sums

    griddep_wait();
    griddep_launch_dependents();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nx = (p.max_q_len + p.TQ - 1) / p.TQ;  // query tiles per (sequence, KV head)
    const int npx = (nx + 1) / 2;                     // pairs of them
    const int n_units = npx * p.H_kv * p.N;
    const int rank = (int)cluster_rank();
    const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;  // this cluster, clusters
    auto slot = [](int i) { return (uint32_t)(i % kWSlots); };
    auto ph = [](int i) { return (uint32_t)((i / kWSlots) & 1); };

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int i = 0; i < kWBars; ++i) mbar_init(sBar + 8 * i, 1);
        for (int b = 0; b < kWSlots; ++b) mbar_init(free0 + 8 * b, 2);  // a slot is free once both CTAs used it
        mbar_init(sfree, kPfSoftmaxThreads);
        mbar_init(prdy, kPfSoftmaxThreads);
        mbar_init(ofree, kPfSoftmaxThreads);
        *abort_flag = 0;
        *armed = 0;
        *armed_q = 0;
        fence_mbar_init();
    }
    // rows past TQ*G (when G does not divide 128) are never loaded: clear them once
    if (warp < 8)
        for (int r = p.TQ * p.G + warp; r < kPfRows; r += 8)
            for (int dh = 0; dh < DH; ++dh)
                if (lane < 8)
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(sQ + dh * kRegion + r * 128 +
                                                                                  lane * 16),
                                 "r"(0)
                                 : "memory");
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // both CTAs' barriers are initialised before either copies or signals into the other
    const uint32_t tmem = *tmem_slot;  // columns: S at 0, O at kWColO, P at kWColP
    auto waited = [&](uint32_t bar, uint32_t parity) {
        const bool w = mbar_wait_bounded(bar, parity, abort_flag, p.wait_ns);
        if (!w) *abort_flag = 1;
        return w;
    };
    bool ok = true;
    WideUnit u;

    if (warp == 8) {
        // ------------------------------------------------------------ TMA producer
        // K and V of a (sequence, KV head) serve every query tile of the row, which neighbouring CTAs run at the
        // same time: kept in L2 (evict_last); a query tile is read once (evict_first)
        const uint64_t pol = policy_evict_last();
        int k = 0, item = 0;  // units and ring items of this CTA so far
        // lane b: the physical block of the tile's b-th KV block, kept per tile parity (V_j is issued after K_{j+1})
        // in two registers
        int ent_even = 0, ent_odd = 0;
        for (int w = cid; w < n_units && ok; w += ncl) {
            const int st = wide_unit<kBf16>(p, nx, npx, w, rank, u);
            if (st == kUnitBadCtx && lane == 0) flag_error(p.err, PA_DEV_ERR_CTX);
            if (st != kUnitOk) continue;
            // the query buffer is free once the previous unit's last S product has completed
            if (k > 0) ok = waited(qfree, (uint32_t)((k - 1) & 1));
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (lane == 0) {
                *armed_q = k + 1;
                mbar_arrive_expect_tx(qbar, (uint32_t)DH * p.G * p.TQ * 128);
                for (int dh = 0; dh < DH; ++dh)
                    tma_load_4d(sQ + dh * kRegion, &tm_q, qbar, 0, dh, u.g * p.G, u.qs + u.tok0, policy_evict_first());
            }
            __syncwarp();
            const int nitems = 2 * u.ntiles;
            for (int i = 0; i < nitems && ok; ++i) {
                int which, t;
                wide_item(i, u.ntiles, which, t);
                const int k0 = t * kWKeys;
                const int nblk = min(kWKeys, u.ctx - k0 + p.B - 1) / p.B;  // blocks holding keys of this tile
                if (which == 0) {
                    int e = lane < nblk ? p.tables[(size_t)u.s * p.MB + k0 / p.B + lane] : 0;
                    if (lane < nblk && (unsigned)e >= (unsigned)p.NB) {
                        flag_error(p.err, PA_DEV_ERR_BLOCK);
                        e = p.NB;  // past the tensor: TMA fills zeros
                    }
                    if (t & 1)
                        ent_odd = e;
                    else
                        ent_even = e;
                }
                const int gi = item + i;
                const uint32_t b = slot(gi);
                // slot b is free once the products of both CTAs that read item gi - kWSlots have completed (either
                // CTA's copies write the slot in both)
                if (gi >= kWSlots) ok = waited(free0 + 8 * b, ph(gi - kWSlots));
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                const uint32_t bar = full0 + 8 * b, dst = sR + b * kSlot;
                // Each CTA copies half of the tile into both CTAs' slot (multicast) and expects the whole tile's bytes
                // on its own barrier; the other half may land before this CTA arms it (the phase cannot complete
                // before the arrival below).
                if (which == 1 && kBf16) {
                    // the staged V tile: 256 keys of this (sequence, KV head); rank r copies keys 128 r .. + 127
                    if (lane == 0) {
                        *armed = gi + 1;
                        mbar_arrive_expect_tx(bar, kSlot);
                        tma_load_5d_mc(dst + (uint32_t)rank * (kSlot / 2), &tm_vsg, bar, 0, 0, 0,
                                       (k0 + rank * kPfKeys) / 8, u.s * p.H_kv + u.g, 0x3, pol);
                    }
                    __syncwarp();
                    continue;
                }
                if (lane == 0) {
                    *armed = gi + 1;  // expect_tx and every copy below, with no wait in between
                    mbar_arrive_expect_tx(bar, (uint32_t)nblk * DH * p.B * 128);
                }
                __syncwarp();
                const int e = (t & 1) ? ent_odd : ent_even;
                if (lane < nblk && (lane & 1) == rank)  // rank r copies the blocks b = r (mod 2)
                    tma_load_5d_mc(dst + (uint32_t)lane * p.B * DH * 128, &tm_kvg, bar, 0, 0, 0, e * (p.B / 8),
                                   which * p.H_kv + u.g, 0x3, pol);
            }
            item += nitems;
            ++k;
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------ MMA issuer
        const uint64_t dq = umma_desc(sQ, 16, 1024);
        auto issue_s = [&](int gi, bool last) {  // S = Q K^T, K (K-major, kGroup bytes per 8 rows) from ring item gi
            const uint64_t dk = umma_desc(sR + slot(gi) * kSlot, 16, kGroup);
#pragma unroll
            for (int ks = 0; ks < NK; ++ks) {
                const uint32_t qoff = (ks >> 2) * (kRegion >> 4) + (ks & 3) * 2;
                const uint32_t koff = (ks >> 2) * (1024 >> 4) + (ks & 3) * 2;
                umma_f16(tmem, dq + qoff, dk + koff, idesc_s, ks > 0);
            }
            umma_commit(sfull);
            umma_commit_mc(free0 + 8 * slot(gi), 0x3);  // both CTAs' slot: either may copy the next item into it
            if (last) umma_commit(qfree);              // the unit's last use of Q
        };
        auto issue_pv = [&](int gi, bool first) {  // O += P V, P from TMEM, V (MN-major, halves 1 KB apart) from gi
            const uint64_t dv = umma_desc(sR + slot(gi) * kSlot, 1024, kGroup);
#pragma unroll
            for (int ks = 0; ks < NT; ++ks)
                umma_f16_ta(tmem + kWColO, tmem + kWColP + ks * 8, dv + (uint64_t)(ks * ((2 * kGroup) >> 4)), idesc_o,
                            (!first || ks > 0));
            umma_commit(pvd);
            umma_commit_mc(free0 + 8 * slot(gi), 0x3);
        };
        if (lane == 0) {
            int k = 0, kt = 0, item = 0;  // units, key tiles and ring items of this CTA so far
            for (int w = cid; w < n_units && ok; w += ncl) {
                if (wide_unit<kBf16>(p, nx, npx, w, rank, u) != kUnitOk) continue;
                const int nt = u.ntiles;
                // S_0 overwrites the previous unit's last S once the softmax has read it, after Q and K_0 landed
                ok = (kt == 0 || waited(sfree, (uint32_t)((kt - 1) & 1))) && waited(qbar, (uint32_t)(k & 1)) &&
                     waited(full0 + 8 * slot(item), ph(item));
                if (!ok) break;
                tc_fence_after();
                issue_s(item, nt == 1);
                for (int j = 0; j < nt && ok; ++j) {
                    if (j + 1 < nt) {
                        const int ik = item + 1 + 2 * j;  // K_{j+1}: S_{j+1} overwrites S_j once the softmax read it
                        ok = waited(sfree, (uint32_t)((kt + j) & 1)) && waited(full0 + 8 * slot(ik), ph(ik));
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(ik, j + 2 == nt);
                    }
                    const int iv = item + (j + 1 < nt ? 2 + 2 * j : 2 * nt - 1);  // V_j
                    // PV_0 starts O afresh: the softmax has read the previous unit's O
                    ok = waited(prdy, (uint32_t)((kt + j) & 1)) && (j > 0 || k == 0 ||
                                                                   waited(ofree, (uint32_t)((k - 1) & 1))) &&
                         waited(full0 + 8 * slot(iv), ph(iv));
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(iv, j == 0);
                }
                kt += nt;
                item += 2 * nt;
                ++k;
            }
            // arrives once every product issued above has completed (at once when none was issued)
            umma_commit(mmadone);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax: thread = (query row, key half)
        const int h = warp >> 2;               // key columns 128 h .. 128 h + 127 of every tile
        const int r = (warp & 3) * 32 + lane;  // query row = TMEM lane
        const uint32_t pair = 1 + (warp & 3);  // named barrier of the two warps holding rows r
        const uint32_t t_lane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t t_s = t_lane + (uint32_t)h * kPfKeys;
        const uint32_t t_p = t_lane + kWColP + (uint32_t)h * (kPfKeys / 2);
        const uint32_t t_o = t_lane + kWColO + (uint32_t)h * (D / 2);
        const float NEG_INF = -INFINITY;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        int kt = 0, item = 0;  // key tiles and ring items of this CTA so far
        bool stop = false;
        for (int w = cid; w < n_units && !stop; w += ncl) {
            if (wide_unit<kBf16>(p, nx, npx, w, rank, u) != kUnitOk) continue;
            const int nt = u.ntiles;
            const int qtok = r / p.G;
            const bool row_ok = r < p.TQ * p.G && u.tok0 >= 0 && u.tok0 + qtok < u.q_len;
            const int qpos = row_ok ? u.pos0 + qtok : -1;  // -1 masks every key
            float m_ref = NEG_INF, l = 0.f;
            for (int j = 0; j < nt; ++j) {
                const int Tj = kt + j;
                const int k0 = j * kWKeys + h * kPfKeys;  // this half's first key
                ok = waited(sfull, (uint32_t)(Tj & 1)) && ok;
                tc_fence_after();
                float v[kPfKeys];
                {
                    uint32_t* uu = reinterpret_cast<uint32_t*>(v);
#pragma unroll
                    for (int c = 0; c < kPfKeys / 32; ++c)
                        asm volatile(
                            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
                            "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
                            "%28, %29, %30, %31}, [%32];"
                            : "=r"(uu[32 * c + 0]), "=r"(uu[32 * c + 1]), "=r"(uu[32 * c + 2]), "=r"(uu[32 * c + 3]),
                              "=r"(uu[32 * c + 4]), "=r"(uu[32 * c + 5]), "=r"(uu[32 * c + 6]), "=r"(uu[32 * c + 7]),
                              "=r"(uu[32 * c + 8]), "=r"(uu[32 * c + 9]), "=r"(uu[32 * c + 10]), "=r"(uu[32 * c + 11]),
                              "=r"(uu[32 * c + 12]), "=r"(uu[32 * c + 13]), "=r"(uu[32 * c + 14]),
                              "=r"(uu[32 * c + 15]), "=r"(uu[32 * c + 16]), "=r"(uu[32 * c + 17]),
                              "=r"(uu[32 * c + 18]), "=r"(uu[32 * c + 19]), "=r"(uu[32 * c + 20]),
                              "=r"(uu[32 * c + 21]), "=r"(uu[32 * c + 22]), "=r"(uu[32 * c + 23]),
                              "=r"(uu[32 * c + 24]), "=r"(uu[32 * c + 25]), "=r"(uu[32 * c + 26]),
                              "=r"(uu[32 * c + 27]), "=r"(uu[32 * c + 28]), "=r"(uu[32 * c + 29]),
                              "=r"(uu[32 * c + 30]), "=r"(uu[32 * c + 31])
                            : "r"(t_s + c * 32)
                            : "memory");
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                }
                tc_fence_before();
                mbar_arrive(sfree);  // S is in registers: the next S product may overwrite it
                // only tiles that reach past the query tile's first position need the causal mask
                if (k0 + kPfKeys - 1 > u.pos0 || !row_ok) {
#pragma unroll
                    for (int i = 0; i < kPfKeys; ++i) v[i] = k0 + i <= qpos ? v[i] : NEG_INF;
                }
                float mx[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
                for (int i = 0; i < kPfKeys; i += 8) {
                    mx[0] = fmax3(mx[0], v[i], v[i + 1]);
                    mx[1] = fmax3(mx[1], v[i + 2], v[i + 3]);
                    mx[2] = fmax3(mx[2], v[i + 4], v[i + 5]);
                    mx[3] = fmax3(mx[3], v[i + 6], v[i + 7]);
                }
                const float m_loc = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * p.scale_log2;  // this half's maximum
                // One barrier per tile as a rule, between the two warps of these rows: it tells both whether a wait
                // gave up, or whether in any of their rows either half's maximum outgrew the reference by more than
                // 2^8.  Only then do the halves of each row exchange their maxima through shared memory (a second
                // barrier, which carries the abort too: the pair leaves at the same barrier, and the other pairs
                // find the abort flag at their next wait).  Otherwise both halves keep the reference, as the
                // exchange would have decided.
                float m_tile = m_loc;
                if (pair_sync_any(pair, j == 0 || m_loc > m_ref + 8.f || !ok || *abort_flag)) {
                    xrow[h * kPfRows + r] = m_loc;
                    if (pair_sync_any(pair, !ok || *abort_flag)) {
                        ok = false;
                        stop = true;
                        break;
                    }
                    m_tile = fmaxf(xrow[r], xrow[kPfRows + r]);
                }
                // both halves of a row take the same decisions from the same values
                float m_new = m_ref;
                if (j == 0 || m_tile > m_ref + 8.f) m_new = fmaxf(m_ref, m_tile);
                const float alpha = (j == 0 || m_new == m_ref) ? 1.f : fast_exp2(m_ref - m_new);
                m_ref = m_new;
                const float m_use = m_new == NEG_INF ? 0.f : m_new;
                const float2 nm2 = make_float2(-m_use, -m_use);
                float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                uint32_t pk[kPfKeys / 2];
#pragma unroll
                for (int i = 0; i < kPfKeys; i += 2) {
                    float2 x = ffma2(make_float2(v[i], v[i + 1]), sc2, nm2);
                    x.x = fast_exp2(x.x);
                    x.y = fast_exp2(x.y);
                    ls[(i >> 1) & 1] = fadd2(ls[(i >> 1) & 1], x);
                    pk[i / 2] = Mma<__half>::pack(x.x, x.y);
                }
                const float2 lsum = fadd2(ls[0], ls[1]);
                l = fmaf(l, alpha, lsum.x + lsum.y);
                // P takes the previous P's columns, and a rescale of O must see the previous PV: both wait for it
                if (Tj > 0) {
                    ok = waited(pvd, (uint32_t)((Tj - 1) & 1)) && ok;
                    tc_fence_after();
                    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                        for (int c = 0; c < D / 64; ++c) {
                            float o[32];
                            tmem_ld32(t_o + c * 32, o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= alpha;
                            tmem_st32(t_o + c * 32, o);
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < kPfKeys / 32; ++c) {
                    uint32_t w16[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w16[i] = pk[16 * c + i];
                    tmem_st16(t_p + c * 16, w16);
                }
                // V rows past the context may hold anything (even NaN) in a tile read from the pool: they are zeroed
                // before PV meets them with P = 0 (a staged tile has zeros there already)
                const int nvalid = min(kWKeys, u.ctx - j * kWKeys);
                if (nvalid < kWKeys && !kBf16) {
                    const int iv = item + (j + 1 < nt ? 2 + 2 * j : 2 * nt - 1);
                    ok = waited(full0 + 8 * slot(iv), ph(iv)) && ok;
                    const uint32_t vb = sR + slot(iv) * kSlot;
                    for (int rr = nvalid + warp; rr < kWKeys; rr += 8)
                        for (int dh = 0; dh < DH; ++dh)
                            if (lane < 8)
                                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(
                                                 vb + (uint32_t)(rr >> 3) * kGroup + dh * 1024 + (rr & 7) * 128 +
                                                 lane * 16),
                                             "r"(0)
                                             : "memory");
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(prdy);
            }
            if (stop) break;
            // the row's exponential sum: this half's plus the other's
            pair_sync(pair);
            xrow[h * kPfRows + r] = l;
            pair_sync(pair);
            const float l_row = xrow[r] + xrow[kPfRows + r];
            if (ok) ok = waited(pvd, (uint32_t)((kt + nt - 1) & 1));
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
                const float inv = 1.f / l_row;
                const size_t orow =
                    ((size_t)(u.qs + u.tok0 + qtok) * p.H_q + (size_t)u.g * p.G + (r % p.G)) * D + h * (D / 2);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    float o[32];
                    tmem_ld32(t_o + c * 32, o);
                    if (c == D / 64 - 1) {
                        tc_fence_before();
                        mbar_arrive(ofree);  // O is read: the next unit's first value product may start it afresh
                    }
                    if (!row_ok) continue;
                    if (p.out_dtype == PA_F32) {
                        // 256-bit stores: each lane writes whole 32-byte sectors of its row (the host checks that
                        // `out` is 32-byte aligned; rows are D floats long)
                        float* dst = static_cast<float*>(p.out) + orow + c * 32;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + 8 * i),
                                         "f"(o[8 * i] * inv), "f"(o[8 * i + 1] * inv), "f"(o[8 * i + 2] * inv),
                                         "f"(o[8 * i + 3] * inv), "f"(o[8 * i + 4] * inv), "f"(o[8 * i + 5] * inv),
                                         "f"(o[8 * i + 6] * inv), "f"(o[8 * i + 7] * inv)
                                         : "memory");
                    } else {
                        T* dst = static_cast<T*>(p.out) + orow + c * 32;
#pragma unroll
                        for (int i = 0; i < 32; ++i) dst[i] = from_float<T>(o[i] * inv);
                    }
                }
            } else {
                mbar_arrive(ofree);
            }
            kt += nt;
            item += 2 * nt;
        }
    }
    // Nothing issued may still be running when TMEM and shared memory are released: the products (the MMA
    // thread's last commit, which follows its commits into the other CTA's barriers) and the copies (the last query
    // tile loaded, each loaded after the previous one was used; and the last arm of each ring slot: slot b's arms
    // are items b, b + 3, ..., each consumed before the next was armed, so only the last can be in flight; its
    // phase completes once both CTAs' halves have landed).  Then the cluster barrier: neither CTA leaves while the
    // other may still copy or signal into it.
    if (warp == 9 && lane == 0) mbar_wait_bounded(mmadone, 0, nullptr);
    if (warp == 8 && lane == 0) {
        const int nq = *armed_q;
        if (nq > 0) mbar_wait_bounded(qbar, (uint32_t)((nq - 1) & 1), nullptr);
        const int n = *armed;
        for (int b = 0; b < kWSlots && b < n; ++b)
            mbar_wait_bounded(full0 + 8 * b, ph(b + (n - 1 - b) / kWSlots * kWSlots), nullptr);
    }
    tc_fence_before();
    ok = __syncthreads_and(ok && !*abort_flag);
    if (!ok && tid == 0) flag_error(p.err, PA_DEV_ERR_TIMEOUT);
    cluster_sync();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ----------------------------------------------------------------------------- host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn pf_encode_fn() {
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

// Which kernel serves the rows with an fp16 value product: prefill_wide_kernel, unless PA_PREFILL_KERNEL=narrow
// (prefill_kernel for every row; =wide names the default).  Measured on the same FLOPs (fp16 / bf16 with V staged,
// TFLOP/s): B = 8: 1122 / 1228 against 1120 / 1064; B = 16: 1335 / 1256 against 1122 / 1048; B = 32: 1314 / 1263
// against 1107 / 1070.  Before its clusters shared each copy, the wide kernel lost at B = 8 (fp16 819).
static bool prefill_use_wide() {
    const char* v = std::getenv("PA_PREFILL_KERNEL");
    return !(v != nullptr && std::strcmp(v, "narrow") == 0);
}

static size_t prefill_smem_bytes(int D) {
    const int DH = D / 64;
    return 1024 + (size_t)(2 + 2 * kPfStages) * DH * kRegion + 256;  // Q[2], K[NS], V[NS], barriers
}

bool prefill_workspace_layout(int N, int H_kv, int D, int B, int MB, PrefillWorkspace* L) {
    if (N <= 0 || H_kv <= 0 || (D != 64 && D != 128) || B <= 0 || MB <= 0) return false;
    const long long keys = (long long)MB * B;
    L->S_pad = (int)((keys + kStagePad - 1) / kStagePad * kStagePad);
    const size_t stage = (size_t)N * H_kv * L->S_pad * D * 2;
    L->split = (stage + 255) & ~size_t(255);
    L->total = L->split + (((size_t)N * H_kv * sizeof(int) + 255) & ~size_t(255));
    return true;
}

template <typename T, int D>
static pa_status run_prefill(const PrefillArgs& a, const CUtensorMap& tq, const CUtensorMap& tkv,
                             const CUtensorMap& tkv_blk, const CUtensorMap& tvs, const CUtensorMap* tvall,
                             const CUtensorMap* tkvg, const CUtensorMap* tvsg, const PrefillWorkspace* ws) {
    auto kern = prefill_kernel<T, D>;
    const size_t smem = prefill_smem_bytes(D);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill)");
    PrefillParams p;
    p.tables = a.tables;
    p.ctx_lens = a.ctx_lens;
    p.q_start = a.q_start;
    p.N = a.N;
    p.T = a.T;
    p.H_q = a.H_q;
    p.H_kv = a.H_kv;
    p.G = a.H_q / a.H_kv;
    p.TQ = kPfRows / p.G;
    p.B = a.B;
    p.MB = a.MB;
    p.NB = a.NB;
    p.out = a.out;
    p.out_dtype = a.out_dtype;
    p.scale_log2 = (float)((double)a.scale * 1.4426950408889634);
    p.wait_ns = wait_limit_ns();
    p.vstage = ws ? a.workspace : nullptr;
    int* vsplit = ws ? reinterpret_cast<int*>(static_cast<uint8_t*>(a.workspace) + ws->split) : nullptr;
    p.vsplit = vsplit;
    p.S_pad = ws ? ws->S_pad : 0;
    p.only_split = 0;
    p.max_q_len = a.max_q_len;
    p.err = a.dev_err;
    if (ws) {
        // stage V as fp16 (before the prefill kernel, same stream); the rows it marks start unmarked
        e = cudaMemsetAsync(vsplit, 0, sizeof(int) * (size_t)a.N * a.H_kv, a.stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync (prefill workspace)");
        const int hb = std::min(kStageHeads, a.H_kv);
        const size_t vsmem = (size_t)kGroupKeys * D * 2 * hb;
        e = cudaFuncSetAttribute(stage_v_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)vsmem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(stage_v)");
        const dim3 sgrid(ws->S_pad / kGroupKeys, (a.H_kv + kStageHeads - 1) / kStageHeads, a.N);
        e = launch_kernel(stage_v_kernel<D>, sgrid, dim3(kStageThreads), vsmem, a.stream, *tvall, a.tables,
                          a.ctx_lens, a.H_kv, a.B, a.MB, a.NB, ws->S_pad, static_cast<uint16_t*>(a.workspace), vsplit,
                          p.wait_ns, a.dev_err);
        count_launch();
        if (e != cudaSuccess) return cuda_fail(e, "V staging launch");
    }
    // fp16 caches and staged bf16 rows: prefill_wide_kernel (fp16 P); bf16 rows without staging, or marked by it:
    // prefill_kernel with the split P (launched after the wide kernel, it serves only the marked rows)
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    if ((!kBf16 || ws) && prefill_use_wide()) {
        auto wide = prefill_wide_kernel<T, D>;
        constexpr size_t wsmem = wide_smem_bytes<D>();
        e = cudaFuncSetAttribute(wide, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)wsmem);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(prefill wide)");
        // persistent: as many 2-CTA clusters as fit at once (one CTA per SM: the shared memory allows no second),
        // at most one per unit (pair of query tiles)
        static std::atomic<int> max_clusters[64];  // per device, per instantiation; 0 = not yet asked
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
        int ncl = max_clusters[dev].load(std::memory_order_relaxed);
        if (ncl == 0) {
            cudaLaunchConfig_t occ = {};
            occ.gridDim = dim3(2);
            occ.blockDim = dim3(kPfThreads);
            occ.dynamicSmemBytes = wsmem;
            int n = 0, per_sm = 0;
            e = cudaOccupancyMaxActiveClusters(&n, wide, &occ);
            if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveClusters(prefill wide)");
            // Each CTA allocates all 512 TMEM columns and keeps them for the whole (persistent) kernel: a second CTA
            // on the same SM would wait in tcgen05.alloc, and with cluster partners waiting on each other that can
            // close a cycle.  Registers (320 threads x 168) allow one CTA per SM; anything else is not launched.
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, wide, kPfThreads, wsmem);
            if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(prefill wide)");
            ncl = (n > 0 && per_sm == 1) ? n : -1;
            max_clusters[dev].store(ncl, std::memory_order_relaxed);
        }
        const long long nx = ((long long)a.max_q_len + p.TQ - 1) / p.TQ;
        const long long units = (nx + 1) / 2 * a.H_kv * a.N;  // the kernel counts units in int
        // otherwise (no 2-CTA cluster fits, or more units than an int counts) every row goes to prefill_kernel
        if (ncl > 0 && units < (1LL << 31)) {
            const dim3 wgrid((unsigned)(2 * std::min<long long>(units, ncl)));
            e = launch_kernel(wide, wgrid, dim3(kPfThreads), wsmem, a.stream, tq, *tkvg, *tvsg, p);
            count_launch();
            if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
            if (!kBf16) return PA_OK;
            p.only_split = 1;
        }
    }
    const dim3 grid((a.max_q_len + 2 * p.TQ - 1) / (2 * p.TQ), a.H_kv, a.N);
    e = launch_kernel(kern, grid, dim3(kPfThreads), smem, a.stream, tq, tkv, tkv_blk, tvs, p);
    count_launch();
    return e == cudaSuccess ? PA_OK : cuda_fail(e, "prefill launch");
}

pa_status launch_prefill(const PrefillArgs& a) {
    EncodeTiledFn fn = pf_encode_fn();
    if (!fn) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int DH = a.D / 64, G = a.H_q / a.H_kv, TQ = kPfRows / G;
    const CUtensorMapDataType dt =
        a.kv_dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUtensorMap tq, tkv;
    std::memset(&tq, 0, sizeof tq);
    std::memset(&tkv, 0, sizeof tkv);
    // queries [T][H_q][D]: dims 64 columns, column half, head, token; box = G heads x TQ tokens
    cuuint64_t qd[4] = {64, (cuuint64_t)DH, (cuuint64_t)a.H_q, (cuuint64_t)a.T};
    cuuint64_t qs[3] = {128, (cuuint64_t)a.D * 2, (cuuint64_t)a.H_q * a.D * 2};
    cuuint32_t qb[4] = {64, 1, (cuuint32_t)G, (cuuint32_t)TQ};
    CUresult r = fn(&tq, dt, 4, const_cast<void*>(a.q), qd, qs, qb, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(q) failed (CUresult %d)", (int)r);
    // pool [NB][B][2][H_kv][D]: dims 64 columns, token, column half, kv head, K/V; box = one block, one half
    cuuint64_t pd[5] = {64, (cuuint64_t)a.NB * a.B, (cuuint64_t)DH, (cuuint64_t)a.H_kv, 2};
    cuuint64_t ps[4] = {(cuuint64_t)2 * a.H_kv * a.D * 2, 128, (cuuint64_t)a.D * 2, (cuuint64_t)a.H_kv * a.D * 2};
    cuuint32_t pb[5] = {64, (cuuint32_t)a.B, 1, 1, 1};
    r = fn(&tkv, dt, 5, const_cast<void*>(a.pool), pd, ps, pb, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(pool) failed (CUresult %d)", (int)r);
    // the same view, box = one whole block (both column halves)
    CUtensorMap tkv_blk;
    std::memset(&tkv_blk, 0, sizeof tkv_blk);
    pb[2] = (cuuint32_t)DH;
    r = fn(&tkv_blk, dt, 5, const_cast<void*>(a.pool), pd, ps, pb, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(pool blocks) failed (CUresult %d)", (int)r);
    // staged V (bf16 caches with a workspace): [N * H_kv][S_pad][D] 16-bit; dims 64 columns, column half, key,
    // (sequence, kv head); box = 128 keys of one half
    CUtensorMap tvs;
    std::memset(&tvs, 0, sizeof tvs);
    PrefillWorkspace ws;
    const bool use_ws = a.kv_dtype == PA_BF16 && a.workspace != nullptr;
    if (use_ws) {
        if (!prefill_workspace_layout(a.N, a.H_kv, a.D, a.B, a.MB, &ws))
            return fail(PA_ERR_INVALID, "invalid prefill workspace arguments");
        if (a.ws_bytes < ws.total) return fail(PA_ERR_INVALID, "prefill workspace too small: %zu < %zu", a.ws_bytes,
                                               ws.total);
        cuuint64_t vd[4] = {64, (cuuint64_t)DH, (cuuint64_t)ws.S_pad, (cuuint64_t)a.N * a.H_kv};
        cuuint64_t vs[3] = {128, (cuuint64_t)a.D * 2, (cuuint64_t)ws.S_pad * a.D * 2};
        cuuint32_t vb[4] = {64, 1, (cuuint32_t)kPfKeys, 1};
        r = fn(&tvs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, a.workspace, vd, vs, vb, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(staged V) failed (CUresult %d)", (int)r);
    }
    // the pool's V rows of up to kStageHeads KV heads of one block, unswizzled, for the staging kernel
    CUtensorMap tvall;
    std::memset(&tvall, 0, sizeof tvall);
    if (use_ws) {
        cuuint32_t vb[5] = {64, (cuuint32_t)a.B, (cuuint32_t)DH, (cuuint32_t)std::min(kStageHeads, a.H_kv), 1};
        r = fn(&tvall, dt, 5, const_cast<void*>(a.pool), pd, ps, vb, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(pool V rows) failed (CUresult %d)", (int)r);
    }
    // prefill_wide_kernel's views: a slot holds [8-row group][column half][8 rows][64 columns].  The pool: dims 64
    // columns, token within a group of 8, column half, group of 8 tokens (over all blocks), K/V x kv head; box = one
    // block.  The staged V: dims 64 columns, key within a group, column half, group of 8 keys, (sequence, kv head);
    // box = 128 keys.
    CUtensorMap tkvg, tvsg;
    std::memset(&tkvg, 0, sizeof tkvg);
    std::memset(&tvsg, 0, sizeof tvsg);
    {
        cuuint64_t gd[5] = {64, 8, (cuuint64_t)DH, (cuuint64_t)a.NB * a.B / 8, (cuuint64_t)2 * a.H_kv};
        cuuint64_t gs[4] = {(cuuint64_t)2 * a.H_kv * a.D * 2, 128, (cuuint64_t)8 * 2 * a.H_kv * a.D * 2,
                            (cuuint64_t)a.D * 2};
        cuuint32_t gb[5] = {64, 8, (cuuint32_t)DH, (cuuint32_t)(a.B / 8), 1};
        r = fn(&tkvg, dt, 5, const_cast<void*>(a.pool), gd, gs, gb, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(pool groups) failed (CUresult %d)", (int)r);
    }
    if (use_ws) {
        cuuint64_t vd[5] = {64, 8, (cuuint64_t)DH, (cuuint64_t)ws.S_pad / 8, (cuuint64_t)a.N * a.H_kv};
        cuuint64_t vs[4] = {(cuuint64_t)a.D * 2, 128, (cuuint64_t)8 * a.D * 2, (cuuint64_t)ws.S_pad * a.D * 2};
        cuuint32_t vb[5] = {64, 8, (cuuint32_t)DH, (cuuint32_t)(kPfKeys / 8), 1};
        r = fn(&tvsg, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, a.workspace, vd, vs, vb, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled(staged V groups) failed (CUresult %d)", (int)r);
    }
    const PrefillWorkspace* w = use_ws ? &ws : nullptr;
    if (a.kv_dtype == PA_BF16)
        return a.D == 128 ? run_prefill<__nv_bfloat16, 128>(a, tq, tkv, tkv_blk, tvs, &tvall, &tkvg, &tvsg, w)
                          : run_prefill<__nv_bfloat16, 64>(a, tq, tkv, tkv_blk, tvs, &tvall, &tkvg, &tvsg, w);
    return a.D == 128 ? run_prefill<__half, 128>(a, tq, tkv, tkv_blk, tvs, &tvall, &tkvg, &tvsg, w)
                      : run_prefill<__half, 64>(a, tq, tkv, tkv_blk, tvs, &tvall, &tkvg, &tvsg, w);
}

}  // namespace pa

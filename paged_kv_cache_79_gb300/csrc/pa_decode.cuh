// Paged decode attention kernels (sm_103a).
//
// Method: "Efficient Memory Management for LLM Serving with PagedAttention"
// (azimuth.plus summary), section "The PagedAttention algorithm": for every block j
// of a sequence the kernel forms s_ji = q.K_ji * scale, the block maximum, the
// block exp-sum and the exp-weighted sum of V, and merges blocks with the
// log-sum-exp rule of the block-wise attention equation (the running-max form of
// the section "Inside: block-table lookup").  The same rule merges the partial
// results of the split-KV partitions in pa_merge_kernel.
//
// Work decomposition.  A work item is (sequence, partition of `partition_blocks`
// blocks, kv head, group of <= 16 query heads sharing that kv head).  A persistent
// grid of CTAs walks the items with a static stride.  Per CTA:
//   warp 4      producer: reads the block table of the item, and for every block
//               issues TMA tile loads of K and V (box = head_dim x block_size of one
//               kv head, 128-byte swizzle) into a ring of shared-memory stages;
//   warps 0..3  consumers: block g of the CTA's stream goes to warp g % 4; each
//               keeps an online-softmax state (max, exp-sum, weighted V) per query
//               head; at the end of an item the four states are merged through
//               shared memory and written as the final output (single-partition
//               sequence) or as a partial (fp32 output + log2-sum-exp).
// For fp16/bf16 the consumers use mma.sync.m16n8k16 with fp32 accumulation:
// S[16 heads x 8 tokens] = Q K^T, then O[16 heads x 8 dims] += P V, P kept in
// registers (the C fragment of Q K^T is the A fragment of P V).  For fp32 they use
// CUDA-core FMAs (tensor cores would round fp32 to tf32).
#pragma once

#include <cfloat>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pagedkv {

template <typename T, int D, int BS>
struct Cfg {
    static constexpr int kElem = (int)sizeof(T);
    static constexpr int kChunkElems = 128 / kElem;  // elements in one 128-byte swizzle row
    static constexpr int kChunks = D / kChunkElems;  // TMA boxes per tile
    static constexpr int kTileBytes = BS * D * kElem;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = (kStageBytes <= 8192) ? 8 : 4;
    static_assert(kStages % kConsumerWarps == 0, "stages must split evenly over consumers");
    static_assert(D % kChunkElems == 0, "head_dim must be a whole number of 128-byte rows");
};

constexpr int kAccPad = 8;  // floats of padding per merge row (spreads banks)

struct SmemLayout {
    uint32_t acc, ml, q, bars, flag, total;
};

__host__ __device__ inline SmemLayout make_layout(int stages, int stage_bytes, int rows, int D,
                                                  bool q_in_smem)
{
    SmemLayout L;
    uint32_t o = (uint32_t)stages * (uint32_t)stage_bytes;
    L.acc = o;
    o += (uint32_t)(kConsumerWarps * rows * (D + kAccPad) * 4);
    L.ml = o;
    o += kConsumerWarps * kHeadsPerItem * 2 * 4;
    L.q = o;
    if (q_in_smem)
        o += (uint32_t)(kConsumerWarps * kHeadsPerItem * D * 4);
    o = (o + 15u) & ~15u;
    L.bars = o;
    o += 2u * (uint32_t)stages * 8u;
    L.flag = o;
    o += 16u;
    L.total = o + 1024u;  // slack to align the base to 1024 bytes (128-byte swizzle)
    return L;
}

__device__ __forceinline__ int clamp_len(const DecodeParams &p, int s, int bs)
{
    const int t = p.context_lens[s];
    const int cap = p.max_blocks * bs;
    return t < 0 ? 0 : (t > cap ? cap : t);
}

__device__ __forceinline__ int num_parts(const DecodeParams &p, int s, int bs)
{
    const int nb = (clamp_len(p, s, bs) + bs - 1) / bs;
    const int np = (nb + p.partition_blocks - 1) / p.partition_blocks;
    return np > 1 ? np : 1;
}

// Warp-cooperative search: move (seq, base) forward to the sequence that owns
// work item w, where base is the index of that sequence's first item.  Items of
// one sequence: num_parts * num_kv_heads * head_groups.  False once w >= total.
__device__ __forceinline__ bool find_item(const DecodeParams &p, int bs, long long w, int &seq,
                                          long long &base, int lane)
{
    const long long units = (long long)p.num_kv_heads * p.head_groups;
    while (seq < p.num_seqs) {
        const int s = seq + lane;
        const long long c = (s < p.num_seqs) ? (long long)num_parts(p, s, bs) * units : 0;
        long long incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += n;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, s < p.num_seqs && base + incl > w);
        if (hit) {
            const int L = __ffs(hit) - 1;
            base += __shfl_sync(0xffffffffu, incl - c, L);
            seq += L;
            return true;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
        seq += 32;
    }
    return false;
}

struct Item {
    int seq, part, kvh, hg, len, j0, j1, qrow0, rows;
    bool single;
};

__device__ __forceinline__ Item decode_item(const DecodeParams &p, int bs, long long w, int seq,
                                            long long base)
{
    Item it;
    const long long units = (long long)p.num_kv_heads * p.head_groups;
    const long long rem = w - base;
    it.seq = seq;
    it.part = (int)(rem / units);
    const int u = (int)(rem % units);
    it.kvh = u / p.head_groups;
    it.hg = u % p.head_groups;
    it.len = clamp_len(p, seq, bs);
    const int nb = (it.len + bs - 1) / bs;
    it.j0 = it.part * p.partition_blocks;
    it.j1 = min(nb, it.j0 + p.partition_blocks);
    it.qrow0 = it.kvh * p.group + it.hg * kHeadsPerItem;
    it.rows = min(kHeadsPerItem, p.group - it.hg * kHeadsPerItem);
    it.single = num_parts(p, seq, bs) == 1;
    return it;
}

// ---------------------------------------------------------------------------
// Producer warp: block-table lookup and TMA tile loads into the stage ring.
// ---------------------------------------------------------------------------
template <int D, int BS, int kChunks, int kTileBytes, int kStages>
__device__ __forceinline__ void producer_loop(const DecodeParams &p, const CUtensorMap *tk,
                                              const CUtensorMap *tv, uint8_t *ring,
                                              uint64_t *full, uint64_t *empty, volatile int *abort,
                                              int lane)
{
    if (lane == 0) {
        dev::tma_prefetch_desc(tk);
        dev::tma_prefetch_desc(tv);
    }
    int seq = 0;
    long long base = 0;
    uint32_t g = 0;
    bool failed = false;
    for (long long w = blockIdx.x; !failed; w += gridDim.x) {
        if (!find_item(p, BS, w, seq, base, lane) || *abort)
            break;
        const Item it = decode_item(p, BS, w, seq, base);
        const int32_t *row = p.block_tables + (size_t)it.seq * p.max_blocks;
        for (int jb = it.j0; jb < it.j1 && !failed; jb += 32) {
            const int j = jb + lane;
            const int phys = (j < it.j1) ? row[j] : 0;  // one coalesced read per 32 blocks
            const int n = min(32, it.j1 - jb);
            for (int i = 0; i < n; ++i, ++g) {
                const int ph = __shfl_sync(0xffffffffu, phys, i);
                const uint32_t st = g % kStages;
                int ok = 1;
                if (lane == 0)
                    ok = dev::mbar_wait(dev::smem_addr(&empty[st]), ((g / kStages) & 1u) ^ 1u,
                                        kWaitTimeoutNs);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) {
                        atomicOr(p.errors, PA_DEVERR_TIMEOUT_EMPTY);
                        *abort = 1;
                    }
                    failed = true;
                    break;
                }
                if (lane == 0) {
                    const uint32_t fb = dev::smem_addr(&full[st]);
                    dev::mbar_arrive_expect_tx(fb, 2u * kTileBytes);
                    // an entry outside the pool reads zeros (fully out-of-bounds box)
                    const int y = (ph >= 0 && ph < p.num_blocks) ? ph * BS : -BS;
                    const uint32_t kd = dev::smem_addr(ring + (size_t)st * 2 * kTileBytes);
                    const uint32_t vd = kd + kTileBytes;
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        dev::tma_load_4d(kd + c * BS * 128, tk, 0, c, it.kvh, y, fb);
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        dev::tma_load_4d(vd + c * BS * 128, tv, 0, c, it.kvh, y, fb);
                }
            }
        }
    }
    if (failed && lane == 0) {
        // Let the copies already issued land before the CTA's shared memory goes away.
        const uint32_t first = g > kStages ? g - kStages : 0;
        for (uint32_t q = first; q < g; ++q)
            dev::mbar_wait(dev::smem_addr(&full[q % kStages]), (q / kStages) & 1u,
                           kWaitTimeoutNs / 8);
    }
}

// ---------------------------------------------------------------------------
// Merge the four consumer states of one item and store it.
// ---------------------------------------------------------------------------
template <typename T, int D>
__device__ __forceinline__ void finalize_item(const DecodeParams &p, const Item &it,
                                              const float *acc, const float *ml, int rows_cap,
                                              int tid)
{
    constexpr int S = D + kAccPad;
    for (int idx = tid; idx < it.rows * D; idx += 32 * kConsumerWarps) {
        const int r = idx / D;
        const int col = idx - r * D;
        float M = -FLT_MAX;
        bool any = false;
#pragma unroll
        for (int c = 0; c < kConsumerWarps; ++c) {
            const float mc = ml[(c * kHeadsPerItem + r) * 2];
            if (mc != -INFINITY) {
                M = fmaxf(M, mc);
                any = true;
            }
        }
        float L = 0.f, O = 0.f;
        if (any) {
#pragma unroll
            for (int c = 0; c < kConsumerWarps; ++c) {
                const float mc = ml[(c * kHeadsPerItem + r) * 2];
                if (mc != -INFINITY) {
                    const float wgt = exp2f(mc - M);
                    L += wgt * ml[(c * kHeadsPerItem + r) * 2 + 1];
                    O += wgt * acc[(c * rows_cap + r) * S + col];
                }
            }
        }
        const float o = (L > 0.f) ? O / L : 0.f;
        const size_t h = (size_t)it.qrow0 + r;
        if (it.single) {
            reinterpret_cast<T *>(p.out)[((size_t)it.seq * p.num_q_heads + h) * D + col] =
                dev::from_float<T>(o);
        } else {
            const size_t pr = ((size_t)it.seq * p.max_parts + it.part) * p.num_q_heads + h;
            p.part_o[pr * D + col] = o;
            if (col == 0)
                p.part_lse[pr] = (L > 0.f) ? M + log2f(L) : -INFINITY;
        }
    }
}

// ---------------------------------------------------------------------------
// fp16 / bf16 partition kernel: tensor-core consumers.
// ---------------------------------------------------------------------------
template <typename T, int D, int BS>
__global__ void __launch_bounds__(kThreads, 2)
    pa_decode_mma_kernel(const __grid_constant__ DecodeParams p,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v)
{
    using C = Cfg<T, D, BS>;
    constexpr int kCE = C::kChunkElems;
    constexpr int NT = BS / 8;   // score n-tiles of 8 tokens
    constexpr int KS = D / 16;   // k-steps of Q K^T
    constexpr int DT = D / 8;    // output n-tiles of 8 dims
    constexpr int SA = D + kAccPad;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int rows_cap = min(kHeadsPerItem, p.group);
    const SmemLayout lay = make_layout(C::kStages, C::kStageBytes, rows_cap, D, false);
    uint8_t *ring = smem;
    float *macc = reinterpret_cast<float *>(smem + lay.acc);
    float *mml = reinterpret_cast<float *>(smem + lay.ml);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
    uint64_t *empty = full + C::kStages;
    volatile int *abort = reinterpret_cast<volatile int *>(smem + lay.flag);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            dev::mbar_init(dev::smem_addr(&full[s]), 1);
            dev::mbar_init(dev::smem_addr(&empty[s]), 1);
        }
        *abort = 0;
        dev::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        producer_loop<D, BS, C::kChunks, C::kTileBytes, C::kStages>(p, &tmap_k, &tmap_v, ring, full,
                                                                   empty, abort, lane);
        return;
    }

    // ---- consumers ----
    const int r0 = lane >> 2;        // fragment row (query head) and row + 8
    const int cq = (lane & 3) * 2;   // fragment column pair
    const int mi = lane >> 3;        // ldmatrix: which 8x8 matrix this lane addresses
    const int swz = lane & 7;        // 128-byte swizzle: 16-byte unit ^= row % 8
    int seq = 0;
    long long base = 0;
    uint32_t g = 0;
    for (long long w = blockIdx.x;; w += gridDim.x) {
        if (!find_item(p, BS, w, seq, base, lane))
            break;
        const Item it = decode_item(p, BS, w, seq, base);

        // Query fragments (A operand of Q K^T); rows past the group are zero.
        uint32_t qa[KS][4];
        {
            const uint32_t *qw = reinterpret_cast<const uint32_t *>(
                reinterpret_cast<const T *>(p.q) + ((size_t)it.seq * p.num_q_heads + it.qrow0) * D);
            const bool v0 = r0 < it.rows, v1 = r0 + 8 < it.rows;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int c0 = (ks * 16 + cq) >> 1;
                qa[ks][0] = v0 ? __ldg(qw + r0 * (D / 2) + c0) : 0u;
                qa[ks][1] = v1 ? __ldg(qw + (r0 + 8) * (D / 2) + c0) : 0u;
                qa[ks][2] = v0 ? __ldg(qw + r0 * (D / 2) + c0 + 4) : 0u;
                qa[ks][3] = v1 ? __ldg(qw + (r0 + 8) * (D / 2) + c0 + 4) : 0u;
            }
        }
        const bool live0 = r0 < it.rows, live1 = r0 + 8 < it.rows;

        float acc[DT][4];
#pragma unroll
        for (int i = 0; i < DT; ++i)
            acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        float mrow0 = -INFINITY, mrow1 = -INFINITY, lrow0 = 0.f, lrow1 = 0.f;
        bool failed = false;

        for (int j = it.j0; j < it.j1; ++j, ++g) {
            if ((int)(g % kConsumerWarps) != warp)
                continue;
            const uint32_t st = g % C::kStages;
            if (!dev::mbar_wait(dev::smem_addr(&full[st]), (g / C::kStages) & 1u, kWaitTimeoutNs)) {
                if (lane == 0) {
                    atomicOr(p.errors, PA_DEVERR_TIMEOUT_FULL);
                    *abort = 1;
                }
                failed = true;
                break;
            }
            const int valid = min(BS, it.len - j * BS);
            const uint32_t kb = dev::smem_addr(ring + (size_t)st * C::kStageBytes);
            const uint32_t vb = kb + C::kTileBytes;

            // S = Q K^T: K tile rows are tokens, so plain ldmatrix yields the
            // "col" B fragment (k = head dim, n = token).
            float sc[NT][4];
#pragma unroll
            for (int i = 0; i < NT; ++i)
                sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int d = ks * 16 + (mi & 1) * 8;
                const uint32_t colpart = (uint32_t)(d / kCE) * (BS * 128) +
                                         (uint32_t)((((d % kCE) >> 3) ^ swz) << 4);
#pragma unroll
                for (int np = 0; np < NT / 2; ++np) {
                    const int tok = (2 * np + (mi >> 1)) * 8 + (lane & 7);
                    uint32_t b0, b1, b2, b3;
                    dev::ldsm_x4(kb + colpart + tok * 128, b0, b1, b2, b3);
                    dev::Mma<T>::run(sc[2 * np], qa[ks], b0, b1);
                    dev::Mma<T>::run(sc[2 * np + 1], qa[ks], b2, b3);
                }
            }

            // block-local softmax statistics merged into the running state
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const bool ok = nt * 8 + cq + e < valid;
                    sc[nt][e] = ok ? sc[nt][e] * p.scale_log2 : -INFINITY;
                    sc[nt][2 + e] = ok ? sc[nt][2 + e] * p.scale_log2 : -INFINITY;
                    mx0 = fmaxf(mx0, sc[nt][e]);
                    mx1 = fmaxf(mx1, sc[nt][2 + e]);
                }
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(mrow0, mx0), mn1 = fmaxf(mrow1, mx1);
            const float corr0 = exp2f(mrow0 - mn0), corr1 = exp2f(mrow1 - mn1);
            mrow0 = mn0;
            mrow1 = mn1;
            float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float a = live0 ? exp2f(sc[nt][e] - mn0) : 0.f;
                    const float b = live1 ? exp2f(sc[nt][2 + e] - mn1) : 0.f;
                    sc[nt][e] = a;
                    sc[nt][2 + e] = b;
                    ps0 += a;
                    ps1 += b;
                }
            }
            lrow0 = lrow0 * corr0 + ps0;
            lrow1 = lrow1 * corr1 + ps1;
            if (__any_sync(0xffffffffu, corr0 != 1.f || corr1 != 1.f)) {
#pragma unroll
                for (int i = 0; i < DT; ++i) {
                    acc[i][0] *= corr0;
                    acc[i][1] *= corr0;
                    acc[i][2] *= corr1;
                    acc[i][3] *= corr1;
                }
            }

            // O += P V: V tile rows are tokens, so ldmatrix.trans yields the
            // "col" B fragment (k = token, n = head dim).
            const bool partial = valid < BS;
#pragma unroll
            for (int kt = 0; kt < BS / 16; ++kt) {
                uint32_t pa[4];
                pa[0] = dev::Mma<T>::pack(sc[2 * kt][0], sc[2 * kt][1]);
                pa[1] = dev::Mma<T>::pack(sc[2 * kt][2], sc[2 * kt][3]);
                pa[2] = dev::Mma<T>::pack(sc[2 * kt + 1][0], sc[2 * kt + 1][1]);
                pa[3] = dev::Mma<T>::pack(sc[2 * kt + 1][2], sc[2 * kt + 1][3]);
                // stale rows past the context may hold anything (NaN): zero them
                uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
                if (partial) {
                    const int t0 = kt * 16 + cq;
                    mk0 = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
                    mk1 = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
                }
                const int tok = kt * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    const int d = dp * 16 + (mi >> 1) * 8;
                    const uint32_t addr = vb + (uint32_t)(d / kCE) * (BS * 128) + tok * 128 +
                                          (uint32_t)((((d % kCE) >> 3) ^ swz) << 4);
                    uint32_t v0, v1, v2, v3;
                    dev::ldsm_x4_trans(addr, v0, v1, v2, v3);
                    dev::Mma<T>::run(acc[2 * dp], pa, v0 & mk0, v1 & mk1);
                    dev::Mma<T>::run(acc[2 * dp + 1], pa, v2 & mk0, v3 & mk1);
                }
            }
            __syncwarp();
            if (lane == 0)
                dev::mbar_arrive(dev::smem_addr(&empty[st]));
        }
        (void)failed;  // a failed warp has set *abort: the CTA stops after this merge

        // ---- merge the four consumer warps ----
        lrow0 += __shfl_xor_sync(0xffffffffu, lrow0, 1);
        lrow0 += __shfl_xor_sync(0xffffffffu, lrow0, 2);
        lrow1 += __shfl_xor_sync(0xffffffffu, lrow1, 1);
        lrow1 += __shfl_xor_sync(0xffffffffu, lrow1, 2);
        float *mine = macc + warp * rows_cap * SA;
        if (live0) {
#pragma unroll
            for (int i = 0; i < DT; ++i)
                *reinterpret_cast<float2 *>(&mine[r0 * SA + i * 8 + cq]) =
                    make_float2(acc[i][0], acc[i][1]);
        }
        if (live1) {
#pragma unroll
            for (int i = 0; i < DT; ++i)
                *reinterpret_cast<float2 *>(&mine[(r0 + 8) * SA + i * 8 + cq]) =
                    make_float2(acc[i][2], acc[i][3]);
        }
        if ((lane & 3) == 0) {
            mml[(warp * kHeadsPerItem + r0) * 2] = (live0 && lrow0 > 0.f) ? mrow0 : -INFINITY;
            mml[(warp * kHeadsPerItem + r0) * 2 + 1] = lrow0;
            mml[(warp * kHeadsPerItem + r0 + 8) * 2] = (live1 && lrow1 > 0.f) ? mrow1 : -INFINITY;
            mml[(warp * kHeadsPerItem + r0 + 8) * 2 + 1] = lrow1;
        }
        dev::consumer_sync(32 * kConsumerWarps);
        finalize_item<T, D>(p, it, macc, mml, rows_cap, threadIdx.x);
        dev::consumer_sync(32 * kConsumerWarps);
        if (*abort)
            break;
    }
}

// ---------------------------------------------------------------------------
// fp32 partition kernel: CUDA-core consumers (same producer, ring and merge).
// ---------------------------------------------------------------------------
template <int D, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    pa_decode_f32_kernel(const __grid_constant__ DecodeParams p,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v)
{
    using C = Cfg<float, D, BS>;
    constexpr int kCE = C::kChunkElems;  // 32 floats per 128-byte row
    constexpr int NPART = 32 / BS;       // lanes per token in the score phase
    constexpr int DP = D / NPART;        // head dims per lane in the score phase
    constexpr int VEC = D / 32;          // head dims per lane in the P V phase
    constexpr int H = kHeadsPerItem;
    constexpr int SA = D + kAccPad;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int rows_cap = min(kHeadsPerItem, p.group);
    const SmemLayout lay = make_layout(C::kStages, C::kStageBytes, rows_cap, D, true);
    uint8_t *ring = smem;
    float *macc = reinterpret_cast<float *>(smem + lay.acc);
    float *mml = reinterpret_cast<float *>(smem + lay.ml);
    float *qsm = reinterpret_cast<float *>(smem + lay.q);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.bars);
    uint64_t *empty = full + C::kStages;
    volatile int *abort = reinterpret_cast<volatile int *>(smem + lay.flag);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            dev::mbar_init(dev::smem_addr(&full[s]), 1);
            dev::mbar_init(dev::smem_addr(&empty[s]), 1);
        }
        *abort = 0;
        dev::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        producer_loop<D, BS, C::kChunks, C::kTileBytes, C::kStages>(p, &tmap_k, &tmap_v, ring, full,
                                                                   empty, abort, lane);
        return;
    }

    const int t = lane % BS;
    const int part = lane / BS;
    float *qs = qsm + warp * H * D;
    int seq = 0;
    long long base = 0;
    uint32_t g = 0;
    for (long long w = blockIdx.x;; w += gridDim.x) {
        if (!find_item(p, BS, w, seq, base, lane))
            break;
        const Item it = decode_item(p, BS, w, seq, base);
        const float *qg = reinterpret_cast<const float *>(p.q) +
                          ((size_t)it.seq * p.num_q_heads + it.qrow0) * D;
        __syncwarp();
        for (int i = lane; i < H * D; i += 32)
            qs[i] = (i / D < it.rows) ? __ldg(qg + i) : 0.f;
        __syncwarp();

        float acc[H][VEC];
        float mr[H], lr[H];
#pragma unroll
        for (int r = 0; r < H; ++r) {
            mr[r] = -INFINITY;
            lr[r] = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                acc[r][e] = 0.f;
        }
        bool failed = false;
        for (int j = it.j0; j < it.j1; ++j, ++g) {
            if ((int)(g % kConsumerWarps) != warp)
                continue;
            const uint32_t st = g % C::kStages;
            if (!dev::mbar_wait(dev::smem_addr(&full[st]), (g / C::kStages) & 1u, kWaitTimeoutNs)) {
                if (lane == 0) {
                    atomicOr(p.errors, PA_DEVERR_TIMEOUT_FULL);
                    *abort = 1;
                }
                failed = true;
                break;
            }
            const int valid = min(BS, it.len - j * BS);
            const uint8_t *kt = ring + (size_t)st * C::kStageBytes;
            const uint8_t *vt = kt + C::kTileBytes;

            float sc[H];
#pragma unroll
            for (int r = 0; r < H; ++r)
                sc[r] = 0.f;
#pragma unroll 4
            for (int u = 0; u < DP / 4; ++u) {
                const int d = part * DP + u * 4;
                const float4 kv = *reinterpret_cast<const float4 *>(
                    kt + (d / kCE) * (BS * 128) + t * 128 + ((((d % kCE) >> 2) ^ (t & 7)) << 4));
#pragma unroll
                for (int r = 0; r < H; ++r) {
                    if (r < it.rows) {
                        const float4 qv = *reinterpret_cast<const float4 *>(&qs[r * D + d]);
                        sc[r] = fmaf(qv.x, kv.x, sc[r]);
                        sc[r] = fmaf(qv.y, kv.y, sc[r]);
                        sc[r] = fmaf(qv.z, kv.z, sc[r]);
                        sc[r] = fmaf(qv.w, kv.w, sc[r]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < H; ++r) {
                if (r >= it.rows)
                    continue;
                float x = sc[r];
                if (NPART == 2)
                    x += __shfl_xor_sync(0xffffffffu, x, 16);
                x = (t < valid) ? x * p.scale_log2 : -INFINITY;
                float mx = x;
#pragma unroll
                for (int o = BS / 2; o > 0; o >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float mn = fmaxf(mr[r], mx);
                const float corr = exp2f(mr[r] - mn);
                mr[r] = mn;
                const float pr = exp2f(x - mn);
                float ssum = pr;
#pragma unroll
                for (int o = BS / 2; o > 0; o >>= 1)
                    ssum += __shfl_xor_sync(0xffffffffu, ssum, o);
                lr[r] = lr[r] * corr + ssum;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    acc[r][e] *= corr;
                sc[r] = pr;
            }
            // P V: lane owns VEC consecutive head dims; only valid rows are read
            for (int tt = 0; tt < valid; ++tt) {
                float v[VEC];
                if constexpr (VEC == 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(
                        vt + (lane >> 3) * (BS * 128) + tt * 128 + (((lane & 7) ^ (tt & 7)) << 4));
                    v[0] = x.x;
                    v[1] = x.y;
                    v[2] = x.z;
                    v[3] = x.w;
                } else {
                    static_assert(VEC == 2, "head_dim 64 or 128");
                    const float2 x = *reinterpret_cast<const float2 *>(
                        vt + (lane >> 4) * (BS * 128) + tt * 128 +
                        ((((lane & 15) >> 1) ^ (tt & 7)) << 4) + (lane & 1) * 8);
                    v[0] = x.x;
                    v[1] = x.y;
                }
#pragma unroll
                for (int r = 0; r < H; ++r) {
                    if (r < it.rows) {
                        const float pt = __shfl_sync(0xffffffffu, sc[r], tt);
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            acc[r][e] = fmaf(pt, v[e], acc[r][e]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                dev::mbar_arrive(dev::smem_addr(&empty[st]));
        }
        (void)failed;

        float *mine = macc + warp * rows_cap * SA;
#pragma unroll
        for (int r = 0; r < H; ++r) {
            if (r < it.rows) {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    mine[r * SA + lane * VEC + e] = acc[r][e];
                if (lane == 0) {
                    mml[(warp * H + r) * 2] = lr[r] > 0.f ? mr[r] : -INFINITY;
                    mml[(warp * H + r) * 2 + 1] = lr[r];
                }
            }
        }
        dev::consumer_sync(32 * kConsumerWarps);
        finalize_item<float, D>(p, it, macc, mml, rows_cap, threadIdx.x);
        dev::consumer_sync(32 * kConsumerWarps);
        if (*abort)
            break;
    }
}

// ---------------------------------------------------------------------------
// Split-KV merge: out[s][h] = sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M).
// One warp per (sequence, query head); sequences with one partition were
// written by the partition kernel.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(128)
    pa_merge_kernel(const __grid_constant__ DecodeParams p, int block_size)
{
    constexpr int VEC = D / 32;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.y;
    const int h = blockIdx.x * 4 + warp;
    if (h >= p.num_q_heads)
        return;
    const int np = num_parts(p, s, block_size);
    if (np <= 1)
        return;
    const size_t hq = (size_t)p.num_q_heads;
    const float *lse = p.part_lse + (size_t)s * p.max_parts * hq + h;
    float M = -INFINITY;
    for (int i = lane; i < np; i += 32)
        M = fmaxf(M, lse[i * hq]);
    M = dev::warp_max(M);
    float W = 0.f;
    for (int i = lane; i < np; i += 32)
        W += exp2f(lse[i * hq] - M);
    W = dev::warp_sum(W);
    const float *po = p.part_o + ((size_t)s * p.max_parts * hq + h) * D + lane * VEC;
    float acc[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e)
        acc[e] = 0.f;
    int i = 0;
    for (; i + 4 <= np; i += 4) {
        float v[4][VEC], wg[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            wg[u] = exp2f(lse[(i + u) * hq] - M);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                v[u][e] = po[(size_t)(i + u) * hq * D + e];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                acc[e] = fmaf(wg[u], v[u][e], acc[e]);
    }
    for (; i < np; ++i) {
        const float wg = exp2f(lse[i * hq] - M);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            acc[e] = fmaf(wg, po[(size_t)i * hq * D + e], acc[e]);
    }
    T *o = reinterpret_cast<T *>(p.out) + ((size_t)s * hq + h) * D + lane * VEC;
#pragma unroll
    for (int e = 0; e < VEC; ++e)
        o[e] = dev::from_float<T>(acc[e] / W);
}

// ---------------------------------------------------------------------------
// Launch helpers
// ---------------------------------------------------------------------------
template <typename T, int D, int BS>
struct KernelOf {
    static void *get() { return reinterpret_cast<void *>(&pa_decode_mma_kernel<T, D, BS>); }
    static constexpr bool kQSmem = false;
};
template <int D, int BS>
struct KernelOf<float, D, BS> {
    static void *get() { return reinterpret_cast<void *>(&pa_decode_f32_kernel<D, BS>); }
    static constexpr bool kQSmem = true;
};

template <typename T, int D, int BS>
inline size_t smem_bytes_for(int group)
{
    using C = Cfg<T, D, BS>;
    const int rows = group < kHeadsPerItem ? group : kHeadsPerItem;
    return make_layout(C::kStages, C::kStageBytes, rows, D, KernelOf<T, D, BS>::kQSmem).total;
}

int cached_occupancy(void *kernel, int device, size_t smem, size_t max_smem);

template <typename T, int D, int BS>
cudaError_t launch_decode_impl(const DecodeLaunch &L, cudaStream_t stream)
{
    const DecodeParams &p = L.p;
    void *kern = KernelOf<T, D, BS>::get();
    const size_t smem = smem_bytes_for<T, D, BS>(p.group);
    const size_t smem_max = smem_bytes_for<T, D, BS>(kHeadsPerItem);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const int per_sm = cached_occupancy(kern, dev, smem, smem_max);
    if (per_sm <= 0)
        return cudaErrorInvalidConfiguration;
    const long long items = (long long)p.num_seqs * p.max_parts * p.num_kv_heads * p.head_groups;
    long long grid = (long long)per_sm * L.sm_count;
    if (L.grid > 0)
        grid = L.grid;
    if (grid > items)
        grid = items;
    if (grid < 1)
        grid = 1;
    void *args[] = {const_cast<DecodeParams *>(&L.p), const_cast<CUtensorMap *>(&L.tmap_k),
                    const_cast<CUtensorMap *>(&L.tmap_v)};
    e = cudaLaunchKernel(kern, dim3((unsigned)grid), dim3(kThreads), args, smem, stream);
    if (e != cudaSuccess)
        return e;
    if (p.max_parts > 1) {
        dim3 mg((unsigned)((p.num_q_heads + 3) / 4), (unsigned)p.num_seqs);
        pa_merge_kernel<T, D><<<mg, 128, 0, stream>>>(p, BS);
        e = cudaGetLastError();
    }
    return e;
}

template <typename T>
cudaError_t launch_decode_dispatch(const DecodeLaunch &L, cudaStream_t stream)
{
    if (L.head_dim == 128 && L.block_size == 16)
        return launch_decode_impl<T, 128, 16>(L, stream);
    if (L.head_dim == 128 && L.block_size == 32)
        return launch_decode_impl<T, 128, 32>(L, stream);
    if (L.head_dim == 64 && L.block_size == 16)
        return launch_decode_impl<T, 64, 16>(L, stream);
    if (L.head_dim == 64 && L.block_size == 32)
        return launch_decode_impl<T, 64, 32>(L, stream);
    return cudaErrorInvalidValue;
}

template <typename T>
size_t smem_dispatch(int head_dim, int block_size, int group)
{
    if (head_dim == 128 && block_size == 16)
        return smem_bytes_for<T, 128, 16>(group);
    if (head_dim == 128 && block_size == 32)
        return smem_bytes_for<T, 128, 32>(group);
    if (head_dim == 64 && block_size == 16)
        return smem_bytes_for<T, 64, 16>(group);
    if (head_dim == 64 && block_size == 32)
        return smem_bytes_for<T, 64, 32>(group);
    return 0;
}

}  // namespace pagedkv

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
// Work decomposition.  A unit is (sequence, kv head, group of <= 16 query heads
// sharing that kv head); a work item is a range of a unit's blocks.  A persistent
// grid of CTAs takes the items in one of two ways:
//   balanced split (partition_size 0): the units' K/V streams are concatenated and
//               each CTA takes an equal contiguous range of ring stages (each unit
//               also charged a fixed cost), so every CTA moves about the same number
//               of bytes; a unit cut by CTA boundaries leaves partials that the CTA
//               completing the set merges;
//   fixed partitions (partition_size > 0): units are cut every partition_size
//               tokens and CTA c takes items c, c + grid, ...; pa_merge_kernel
//               combines the partitions of multi-partition sequences.
// Per CTA:
//   warp 4      producer: reads the block table of the item, and for every block
//               issues TMA tile loads of K and V (box = head_dim x block_size of one
//               kv head, 128-byte swizzle) into a ring of shared-memory stages;
//   warps 0..3  consumers: ring stage i of an item (32 tokens for fp16/bf16, one
//               block for fp32) goes to warp (i + rot) % 4, rot fixed by the item's
//               place in the stream, so consecutive items continue the rotation and
//               the rounding does not depend on which CTA runs an item; each warp
//               keeps an online-softmax state (max, exp-sum, weighted V) per query
//               row; at the end of an item the four states are merged through
//               shared memory and written as the final output (the item is a whole
//               unit) or as a partial (fp32 output + log2-sum-exp).
// For fp16/bf16 the consumers use mma.sync.m16n8k16 with fp32 accumulation.  Items
// of up to 8 query rows (a group of <= 8 heads, or the members of a shared prefix)
// take the transposed products S^T[tokens x rows] = K Q^T and O^T += V^T P^T, so a
// 16-row MMA tile carries 16 tokens rather than padding rows; wider items take
// S[16 rows x 8 tokens] = Q K^T, then O += P V, P kept in registers (the C fragment
// of Q K^T is the A fragment of P V).  For fp32 they use CUDA-core FMAs (tensor
// cores would round fp32 to tf32).
#pragma once

#include <cfloat>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pagedkv {

#ifndef PA_RING_BYTES
#define PA_RING_BYTES 65536  // shared memory of the stage ring (two CTAs per SM)
#endif

// A ring stage holds the K and V tiles of kBPS consecutive blocks of one item
// (kStageTokens token rows of one kv head): per block its K tile, then its V tile,
// so that one copy can fetch both (tile_at).  A tile is d / (128 bytes) runs of
// BS rows of 128 bytes (chunk-major), 128-byte swizzled.
template <typename T, int D, int BS>
struct Cfg {
    static constexpr int kElem = (int)sizeof(T);
    static constexpr int kChunkElems = 128 / kElem;  // elements in one 128-byte swizzle row
    static constexpr int kChunks = D / kChunkElems;  // 128-byte rows per token row
    static constexpr int kStageTokens =
        (sizeof(T) == 4 || PA_STAGE_TOKENS <= BS) ? BS : PA_STAGE_TOKENS;
    static constexpr int kBPS = kStageTokens / BS;   // blocks per stage
    static constexpr int kTileBytes = kStageTokens * D * kElem;  // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kBlockTile = BS * D * kElem;    // K (or V) of one block
    static constexpr int kBlockStride = 2 * kBlockTile;  // one block's K and V tiles
    static constexpr int kStagesRaw = (PA_RING_BYTES / kStageBytes) / kConsumerWarps * kConsumerWarps;
    static constexpr int kStages = kStagesRaw < kConsumerWarps ? kConsumerWarps : kStagesRaw;
    static_assert(kStages % kConsumerWarps == 0, "stages must split evenly over consumers");
    static_assert(D % kChunkElems == 0, "head_dim must be a whole number of 128-byte rows");
    static_assert(kStageTokens % BS == 0 && 32 % kBPS == 0, "a stage is a whole number of blocks");
};

// Addressing a ring stage: the 128-byte row holding chunk ch (bytes 128 ch ..
// 128 ch + 127 of the head dim) of token t16 + r's K row, for t16 a multiple of 16
// and r < 16, lies at
//     tile_at(t16) + ch * BS * 128 + r * 128        (V: + kBlockTile)
// and its 16-byte units are swizzled by r % 8.  tile_at folds to a constant in the
// consumers' unrolled token loops.  With one block per stage (tile_at(t16) =
// t16 * 128) the narrow consumers address a row as base + chunk term + token * 128,
// the form the stage layout had before it held two blocks: code generated from the
// two-block form measured 0.4% slower on the long-context decode there.
template <int BS, int kBlockStride>
__device__ __forceinline__ constexpr uint32_t tile_at(int t16)
{
    return (uint32_t)((t16 / BS) * kBlockStride + (t16 % BS) * 128);
}

// How the producer copies a block's K and V tiles: one copy through the joint
// tensor map, one copy per cache, or (fp32 kernels) whichever the launch's
// kv_joint says.  The fp16/bf16 kernels are built for the first two, so their
// producer loop carries no test of it.
constexpr int kCopyRuntime = 0;
constexpr int kCopyJoint = 1;
constexpr int kCopySplit = 2;

constexpr int kAccPad = 8;  // floats of padding per merge row (spreads banks)

// Debug builds (-DPA_TRACE) record per-CTA timestamps (ns) and counters into a
// device array read back with pa_debug_trace_<dtype>; normal builds compile the
// hooks away.
#ifdef PA_TRACE
constexpr int kTraceSlots = 16;
constexpr int kTraceCtas = 4096;  // rows: CTA index, plus half the rows for shared pass 1
static __device__ unsigned long long g_trace[kTraceCtas * kTraceSlots];
__device__ __forceinline__ int trace_row(int pass)
{
    const int r = (int)blockIdx.x + (pass ? kTraceCtas / 2 : 0);
    return r < kTraceCtas ? r : -1;
}
// -DPA_TRACE_LITE keeps only the once-per-CTA stamps (start, end, SM, items, first
// item, first tile issued, producer end), whose cost does not distort the schedule
#ifdef PA_TRACE_LITE
constexpr bool kTraceLite = true;
#else
constexpr bool kTraceLite = false;
#endif
// Per-stage and per-item stamps: the stamps-only build reads no timer for them (a
// %globaltimer read per stage slowed the decode by a fifth).
__device__ __forceinline__ unsigned long long trace_clock()
{
    return kTraceLite ? 0ull : dev::global_timer_ns();
}
__device__ __forceinline__ void trace_set(int pass, int slot, unsigned long long v)
{
    const int r = trace_row(pass);
    if (r >= 0 && (!kTraceLite || slot == 0 || slot == 2 || slot == 3 || slot == 4 || slot == 8 || slot >= 14))
        g_trace[r * kTraceSlots + slot] = v;
}
__device__ __forceinline__ void trace_add(int pass, int slot, unsigned long long v)
{
    const int r = trace_row(pass);
    if (r >= 0 && !kTraceLite)
        g_trace[r * kTraceSlots + slot] += v;
}
__device__ __forceinline__ bool trace_first_tile(int pass)
{
    const int r = trace_row(pass);
    return !kTraceLite && r >= 0 && g_trace[r * kTraceSlots + 1] == 0;
}
// call sites have the launch's DecodeParams in scope as `p`
#define PA_TRACE_SET(slot, v) trace_set(p.pass, (slot), (v))
#define PA_TRACE_ADD(slot, v) trace_add(p.pass, (slot), (v))
#define PA_TRACE_DEFINE_READER(name)                                                     \
    extern "C" int pa_debug_trace_##name(unsigned long long *host, int n, int clear)      \
    {                                                                                   \
        int e = (int)cudaMemcpyFromSymbol(host, pagedkv::g_trace, (size_t)n * 8);        \
        if (clear) {                                                                    \
            static unsigned long long zeros[pagedkv::kTraceCtas * pagedkv::kTraceSlots]; \
            cudaMemcpyToSymbol(pagedkv::g_trace, zeros, sizeof zeros);                  \
        }                                                                               \
        return e;                                                                       \
    }
#else
#define PA_TRACE_SET(slot, v)
#define PA_TRACE_ADD(slot, v)
#define PA_TRACE_DEFINE_READER(name)
#endif

struct SmemLayout {
    uint32_t acc, ml, pfx, items, q, newrow, newinfo, bars, flag, blk, total;
};

// Shared-prefix buffer rows: o (head_dim floats), then the log2-sum-exp, padded to
// a multiple of 16 bytes.
constexpr int kPfxPad = 4;

constexpr int kItemSlots = 2;  // work-item descriptors (and their query rows) in flight

constexpr int kNarrowRows = 8;  // items of at most this many rows use the transposed form

// Most query rows one item of this launch carries: the heads of one head group,
// or, in the shared-prefix pass, the rows of up to kHeadsPerItem / group member
// sequences.  Sizes the merge accumulators in shared memory.
__host__ __device__ inline int item_rows_cap(const DecodeParams &p)
{
    if (p.pass == 1)
        return p.group <= kNarrowRows ? kNarrowRows : kHeadsPerItem;
    return p.group < kHeadsPerItem ? p.group : kHeadsPerItem;
}

// Rows of shared-prefix data an item of this launch merges (pass 0 of the
// shared-prefix decode), else 0.
__host__ __device__ inline int item_pfx_rows(const DecodeParams &p)
{
    return (p.pass == 0 && p.share) ? item_rows_cap(p) : 0;
}

// Members of a group whose query rows share one shared-prefix item: the rows
// fill the 8-row (group <= 8) or 16-row item.
__host__ __device__ inline int members_per_item(int group)
{
    return (group <= kNarrowRows ? kNarrowRows : kHeadsPerItem) / group;
}

// Shared memory: stage ring | merge accumulators | merge (max, sum) | shared-prefix
// rows (two item buffers; pass 0 of the shared-prefix decode only) | item
// descriptors | query rows per item slot | mbarriers | flags | the producer's block
// ids.
__host__ __device__ inline SmemLayout make_layout(int stages, int stage_bytes, int rows, int D,
                                                  int elem_bytes, int pfx_rows = 0)
{
    SmemLayout L;
    uint32_t o = (uint32_t)stages * (uint32_t)stage_bytes;
    L.acc = o;
    o += (uint32_t)(kConsumerWarps * rows * (D + kAccPad) * 4);
    L.ml = o;
    o += kConsumerWarps * kHeadsPerItem * 2 * 4;
    o = (o + 127u) & ~127u;
    L.pfx = o;
    o += (uint32_t)(2 * pfx_rows * (D + kPfxPad) * 4);
    L.items = o;
    o += kItemSlots * 64u;
    L.q = o;
    o += (uint32_t)(kItemSlots * kHeadsPerItem * D * elem_bytes);
    L.newrow = o;  // per stage: the newest token's K row then V row (fused append)
    o += (uint32_t)(stages * 2 * D * elem_bytes);
    L.newinfo = o;  // per stage: {row in the stage tile or -1, physical block}
    o += (uint32_t)(stages * 8);
    o = (o + 15u) & ~15u;
    L.bars = o;
    o += (2u * (uint32_t)stages + 2u * kItemSlots + 1u) * 8u;
    L.flag = o;  // abort flag, merge flag, counter seen, then a scratch word per consumer warp
    o += 16u + 4u * kConsumerWarps;
    o = (o + 15u) & ~15u;
    L.blk = o;  // the producer's current window of 32 block ids
    o += 32u * 4u;
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

constexpr int kToPrefix = 1;     // result rows go to the shared-prefix buffer
constexpr int kMergePrefix = 2;  // result rows are merged with the shared-prefix buffer

// Kernel instances by launch: a plain decode carries no shared-prefix code (code
// it never runs still costs a small decode ~2 us); the shared-prefix decode's two
// launches each have their own.
constexpr int kModePlain = 0;   // pa_decode, pa_decode_append
constexpr int kModePrefix = 1;  // shared-prefix decode, pass 1: the groups' shared blocks
constexpr int kModeOwn = 2;     // shared-prefix decode, pass 0: every sequence's own blocks
constexpr int kModePlan = 3;    // pa_decode_planned: the plain decode, each CTA's start planned on the host

// A work item: blocks [j0, j1) of one unit.  Row r of the item is query head
// qrow0 + r % rpm of sequence seq + r / rpm (several sequences only in the
// shared-prefix pass, where the rows of `members` sequences share one kv head).
struct Item {
    int seq, kvh, hg, len;  // first sequence, kv head, head group, context length
    int j0, j1;             // blocks [j0, j1) of the unit (absolute block indices)
    int qrow0, rows;        // query heads qrow0 .. of each sequence; rows in all
    int partial;            // 0: write the result; 1: write partial row prow0 + r
    int prow0;
    // balanced split, partial items: the unit's partials come from the non-empty
    // CTAs c_first ... (nparts of them); the CTA that writes the last one merges
    int c_first, nparts;
    unsigned int total_lo, total_hi;  // stream length (to tell empty CTA ranges)
    int tseq;               // sequence whose block-table row gives the blocks
    int packed;             // members << 16 | rows per member << 8 | divisor << 4 | rot << 2 | flags
    __device__ int members() const { return packed >> 16; }
    __device__ int rpm() const { return (packed >> 8) & 0xff; }
    __device__ int flags() const { return packed & 3; }  // kToPrefix / kMergePrefix
    // Stage i of the item goes to consumer warp (i + rot) % 4.  rot is a function of
    // the item alone (not of the CTA that runs it), so the warps' partial sums, and
    // with them the rounding of the result, do not depend on the schedule.
    __device__ int rot() const { return (packed >> 2) & 3; }
    // balanced split: positions per CTA the stream was cut by (see balanced_divisor)
    __device__ int divisor() const { return (packed >> 4) & 0xf; }
};
static_assert(sizeof(Item) == 64, "one 64-byte descriptor slot");

__device__ __forceinline__ int pack_rows(int members, int rpm, int flags, int rot = 0)
{
    return (members << 16) | (rpm << 8) | ((rot & 3) << 2) | flags;
}

__device__ __forceinline__ Item decode_item(const DecodeParams &p, int bs, long long w, int seq,
                                            long long base)
{
    Item it;
    const long long units = (long long)p.num_kv_heads * p.head_groups;
    const long long rem = w - base;
    it.seq = seq;
    // the kv heads of one partition are adjacent (they share DRAM pages)
    const int part = (int)(rem / units);
    const int u = (int)(rem % units);
    it.kvh = u / p.head_groups;
    it.hg = u % p.head_groups;
    it.len = clamp_len(p, seq, bs);
    const int nb = (it.len + bs - 1) / bs;
    it.j0 = part * p.partition_blocks;
    it.j1 = min(nb, it.j0 + p.partition_blocks);
    it.qrow0 = it.kvh * p.group + it.hg * kHeadsPerItem;
    it.rows = min(kHeadsPerItem, p.group - it.hg * kHeadsPerItem);
    it.partial = num_parts(p, seq, bs) == 1 ? 0 : 1;
    it.prow0 = (int)(((long long)seq * p.max_parts + part) * p.num_q_heads + it.qrow0);
    it.c_first = -1;  // merged by pa_merge_kernel
    it.nparts = 0;
    it.total_lo = it.total_hi = 0;
    it.tseq = seq;
    it.packed = pack_rows(1, it.rows, 0, (int)(w & 3));
    return it;
}

// ---------------------------------------------------------------------------
// Per-CTA shared state.
// ---------------------------------------------------------------------------
struct CtaState {
    uint8_t *ring;
    float *macc;
    float *mml;
    Item *items;
    uint8_t *qslots;
    uint8_t *newrow;                   // per ring stage: fused-append K/V rows
    volatile int *newinfo;             // per ring stage: {row or -1, physical block}
    uint64_t *full, *empty;            // per ring stage
    uint64_t *item_full, *item_empty;  // per item slot
    uint64_t *csync;                   // consumer-only barrier (all consumer threads arrive)
    float *pfx;                        // two buffers of shared-prefix rows (item parity)
    volatile int *abort;
    volatile int *merge;               // this CTA completes the current split unit
    unsigned long long *ctr_seen;      // the split unit's counter as the probe read it
    volatile uint32_t *sink;           // per consumer warp: see dev::settle_loads
    int *blk;                          // the producer's window of 32 block ids
};

__device__ __forceinline__ CtaState cta_state(uint8_t *smem, const SmemLayout &lay, int stages)
{
    CtaState c;
    c.ring = smem;
    c.macc = reinterpret_cast<float *>(smem + lay.acc);
    c.mml = reinterpret_cast<float *>(smem + lay.ml);
    c.items = reinterpret_cast<Item *>(smem + lay.items);
    c.qslots = smem + lay.q;
    c.newrow = smem + lay.newrow;
    c.newinfo = reinterpret_cast<volatile int *>(smem + lay.newinfo);
    c.full = reinterpret_cast<uint64_t *>(smem + lay.bars);
    c.empty = c.full + stages;
    c.item_full = c.empty + stages;
    c.item_empty = c.item_full + kItemSlots;
    c.csync = c.item_empty + kItemSlots;
    c.pfx = reinterpret_cast<float *>(smem + lay.pfx);
    c.abort = reinterpret_cast<volatile int *>(smem + lay.flag);
    c.merge = reinterpret_cast<volatile int *>(smem + lay.flag + 4);
    c.ctr_seen = reinterpret_cast<unsigned long long *>(smem + lay.flag + 8);
    c.sink = reinterpret_cast<volatile uint32_t *>(smem + lay.flag + 16);
    c.blk = reinterpret_cast<int *>(smem + lay.blk);
    return c;
}

__device__ __forceinline__ bool defers_dependency(const DecodeParams &p)
{
    return p.pass == 0 && p.share != nullptr;
}

__device__ __forceinline__ void init_cta(const DecodeParams &p, const CtaState &c, int stages)
{
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            dev::mbar_init(dev::smem_addr(&c.full[s]), 1);
            dev::mbar_init(dev::smem_addr(&c.empty[s]), 1);
        }
        for (int i = 0; i < kItemSlots; ++i) {
            dev::mbar_init(dev::smem_addr(&c.item_full[i]), 1);
            dev::mbar_init(dev::smem_addr(&c.item_empty[i]), kConsumerWarps);
        }
        dev::mbar_init(dev::smem_addr(c.csync), 32 * kConsumerWarps);
        *c.abort = 0;
        dev::fence_mbar_init();
    }
    __syncthreads();
    // Everything read below may be produced by the previous kernel in the stream,
    // except in pass 0 of the shared-prefix decode: the previous kernel is pass 1,
    // which writes only the prefix rows (and its own counters and partial slots),
    // so pass 0 streams its blocks while pass 1 finishes and waits only before it
    // first reads a prefix row (its own predecessors had completed before pass 1
    // passed this point).
    if (!defers_dependency(p))
        dev::grid_dependency_wait();
    dev::grid_launch_dependents();
}

// Copy a descriptor out of its slot.  The volatile reads happen here and only here:
// once the slot is released the producer may overwrite it with a later item, so
// the compiler must not re-read fields from shared memory afterwards.
__device__ __forceinline__ Item load_item(const Item *slot)
{
    const volatile int *v = reinterpret_cast<const volatile int *>(slot);
    Item it;
    it.seq = v[0];
    it.kvh = v[1];
    it.hg = v[2];
    it.len = v[3];
    it.j0 = v[4];
    it.j1 = v[5];
    it.qrow0 = v[6];
    it.rows = v[7];
    it.partial = v[8];
    it.prow0 = v[9];
    it.c_first = v[10];
    it.nparts = v[11];
    it.total_lo = (unsigned int)v[12];
    it.total_hi = (unsigned int)v[13];
    it.tseq = v[14];
    it.packed = v[15];
    return it;
}

__device__ __forceinline__ void raise_error(const DecodeParams &p, volatile int *abort,
                                            unsigned int flag)
{
    atomicOr(p.errors, flag);
    *abort = 1;
}

// Bounded wait on an mbarrier phase by every lane of a consumer warp; warp-uniform
// result.  It gives up after the launch's wait limit and raises
// PA_DEVERR_TIMEOUT_FULL.  (It does not watch the CTA's abort flag: with that
// check in this wait the shared-prefix decode took 221 us instead of 215.  A
// consumer left waiting after another warp gave up runs to its own limit.)
__device__ __forceinline__ bool warp_wait(const DecodeParams &p, const CtaState &c, uint64_t *bar,
                                          uint32_t parity)
{
    const bool ok = __all_sync(0xffffffffu, dev::mbar_wait(dev::smem_addr(bar), parity, p.wait_ns));
    if (!ok && (threadIdx.x & 31) == 0)
        raise_error(p, c.abort, PA_DEVERR_TIMEOUT_FULL);
    return ok;
}

// Barrier among the consumer warps only (the producer runs ahead), bounded.
__device__ __forceinline__ bool consumer_sync(const DecodeParams &p, const CtaState &c,
                                              uint32_t &phase)
{
    dev::mbar_arrive(dev::smem_addr(c.csync));
    const bool ok = warp_wait(p, c, c.csync, phase & 1u);
    ++phase;
    return ok;
}

// ---------------------------------------------------------------------------
// Producer warp: walks the work items, publishes each item's descriptor and
// query rows (one bulk copy) to an item slot, then looks the item's blocks up in
// the block table and issues their K/V TMA tile loads into the stage ring.
// ---------------------------------------------------------------------------
template <typename T, int D, int BS, int kBPS, int kChunks, int kTileBytes, int kStages, int kCopy>
struct Producer {
    const DecodeParams &p;
    const CUtensorMap *tk;
    const CUtensorMap *tv;
    const CtaState &c;
    int lane;
    uint32_t g;  // stages issued
    uint32_t n;  // items published
    bool failed;
    // pa_decode_planned: the block ids of the CTA's first item's first window, one
    // per lane from lane 16 on (kPlanWindow of them); plan_seq < 0 once used
    int plan_blk;
    int plan_seq;
    int plan_j0;
#ifdef PA_TRACE
    unsigned long long t_last_issue;
#endif

    __device__ Producer(const DecodeParams &p_, const CUtensorMap *tk_, const CUtensorMap *tv_,
                        const CtaState &c_, int lane_)
        : p(p_), tk(tk_), tv(tv_), c(c_), lane(lane_), g(0), n(0), failed(false), plan_blk(0),
          plan_seq(-1), plan_j0(0)
    {
#ifdef PA_TRACE
        t_last_issue = 0;
#endif
        if (lane == 0) {
            dev::tma_prefetch_desc(tk);
            dev::tma_prefetch_desc(tv);
        }
    }

    // Publish `it` and stream its blocks; false once the CTA is stopping early (a
    // wait gave up, here or in a consumer warp).
    __device__ bool emit(const Item &it)
    {
        constexpr uint32_t kQSlotBytes = kHeadsPerItem * D * sizeof(T);
        {
            const uint32_t slot = n % kItemSlots;
            int ok = 1;
#ifdef PA_TRACE
            if (lane == 0 && n == 0)
                PA_TRACE_SET(15, dev::global_timer_ns());  // first item found
#endif
            if (lane == 0) {
                ok = wait_slot(&c.item_empty[slot], ((n / kItemSlots) & 1u) ^ 1u);
                if (ok) {
                    c.items[slot] = it;
                    // query rows: rpm contiguous heads of each member sequence
                    const uint32_t mbytes = (uint32_t)it.rpm() * D * sizeof(T);
                    const uint32_t fb = dev::smem_addr(&c.item_full[slot]);
                    dev::mbar_arrive_expect_tx(fb, mbytes * (uint32_t)it.members());
                    for (int m = 0; m < it.members(); ++m)
                        dev::bulk_load(dev::smem_addr(c.qslots + slot * kQSlotBytes) + m * mbytes,
                                       reinterpret_cast<const T *>(p.q) +
                                           ((size_t)(it.seq + m) * p.num_q_heads + it.qrow0) * D,
                                       mbytes, fb);
                }
            }
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                failed = true;
                return false;
            }
            ++n;
        }
        const int32_t *row = p.block_tables + (size_t)it.tseq * p.max_blocks;
        // a planned first item takes its first kPlanWindow block ids from the plan
        // (no block-table round trip before its first copies), then 32 at a time.
        // The warp loads a window of ids into shared memory; lane 0 alone then
        // waits for and fills the window's stages, with no warp-wide step per stage.
        const bool planned = plan_seq == it.tseq && plan_j0 == it.j0;
        plan_seq = -1;
        for (int jb = it.j0, wnd = 32; jb < it.j1; jb += wnd) {
            const bool from_plan = planned && jb == it.j0;
            wnd = from_plan ? kPlanWindow : 32;
            const int j = jb + lane;
            int phys;
            if (from_plan)
                phys = __shfl_sync(0xffffffffu, plan_blk, (lane % kPlanWindow) + kPlanBlocks);
            else
                phys = (j < it.j1) ? row[j] : 0;  // one coalesced read per 32 blocks
            const int cnt = min(wnd, it.j1 - jb);
            c.blk[lane] = phys;
            __syncwarp();
            uint32_t issued = 0;
            int ok = 1;
            if (lane == 0)
                ok = fill_window(it, row, jb, cnt, from_plan, issued);
            // lane 0 has read the window's ids once the warp passes these
            g += __shfl_sync(0xffffffffu, issued, 0);
            if (!__shfl_sync(0xffffffffu, ok, 0)) {
                failed = true;
                return false;
            }
        }
        return true;
    }

    // Lane 0: the stages of one window of cnt blocks (ids in c.blk) starting at block
    // jb of the item.  Returns false once a wait gave up; *issued: stages issued.
    __device__ int fill_window(const Item &it, const int32_t *row, int jb, int cnt,
                               bool from_plan, uint32_t &issued)
    {
        constexpr int kBlockTile = kTileBytes / kBPS;
        constexpr uint32_t kRowBytes = D * sizeof(T);
        uint32_t gg = g;
        for (int i = 0; i < cnt; i += kBPS, ++gg) {
            const int nbs = min(kBPS, cnt - i);  // blocks in this stage
            const uint32_t st = gg % kStages;
            if (!wait_slot(&c.empty[st], ((gg / kStages) & 1u) ^ 1u)) {
                issued = gg - g;
                return 0;
            }
            const uint32_t fb = dev::smem_addr(&c.full[st]);
            // fused append: does this stage hold the sequence's newest token?
            const int newest = it.len - 1 - (jb + i) * BS;
            const bool has_new = p.k_new != nullptr && newest >= 0 && newest < nbs * BS;
            c.newinfo[2 * st] = has_new ? newest : -1;
            // the block the newest token is written to always comes from the
            // table, so a stale plan cannot direct the append elsewhere
            if (has_new)
                c.newinfo[2 * st + 1] =
                    from_plan ? row[jb + i + newest / BS] : c.blk[(i + newest / BS) & 31];
            dev::mbar_arrive_expect_tx(
                fb, 2u * (uint32_t)nbs * kBlockTile + (has_new ? 2u * kRowBytes : 0u));
            if (has_new) {
                const size_t src = ((size_t)it.seq * p.num_kv_heads + it.kvh) * D;
                const uint32_t nr = dev::smem_addr(c.newrow + (size_t)st * 2 * kRowBytes);
                dev::bulk_load(nr, reinterpret_cast<const T *>(p.k_new) + src, kRowBytes, fb);
                dev::bulk_load(nr + kRowBytes, reinterpret_cast<const T *>(p.v_new) + src, kRowBytes,
                               fb);
            }
            const uint32_t kd = dev::smem_addr(c.ring + (size_t)st * 2 * kTileBytes);
#pragma unroll
            for (int b = 0; b < kBPS; ++b) {
                if (b < nbs) {
                    const int id = c.blk[(i + b) & 31];
                    // an entry outside the pool reads zeros (fully out-of-bounds box)
                    const int y = (id >= 0 && id < p.num_blocks) ? id * BS : -BS;
                    const uint32_t dst = kd + (uint32_t)b * 2 * kBlockTile;
                    if (kCopy == kCopyJoint || (kCopy == kCopyRuntime && p.kv_joint)) {
                        dev::tma_load_5d(dst, tk, 0, y, 0, it.kvh, 0, fb);  // K and V
                    } else {
                        dev::tma_load_4d(dst, tk, 0, y, 0, it.kvh, fb);
                        dev::tma_load_4d(dst + kBlockTile, tv, 0, y, 0, it.kvh, fb);
                    }
                }
            }
#ifdef PA_TRACE
            if (!t_last_issue)
                PA_TRACE_SET(14, dev::global_timer_ns());  // first tile issued
            t_last_issue = kTraceLite ? 1ull : dev::global_timer_ns();
            PA_TRACE_ADD(7, 1);
#endif
        }
        issued = gg - g;
        return 1;
    }

    // Lane 0: wait for the consumers to free a ring stage or item slot (the phase
    // before `parity`).  Gives up after the launch's wait limit, raising
    // PA_DEVERR_TIMEOUT_EMPTY, or once a consumer warp has given up.
    __device__ bool wait_slot(uint64_t *bar, uint32_t parity)
    {
        const int r = dev::mbar_wait_abortable(dev::smem_addr(bar), parity, p.wait_ns, c.abort);
        if (r == 0)
            raise_error(p, c.abort, PA_DEVERR_TIMEOUT_EMPTY);
        return r == 1;
    }

    // End of the walk: publish the end-of-work marker for the consumers (unless the
    // CTA is stopping early), and let every copy this warp issued land before it
    // exits.  The CTA's shared memory stays allocated while any of its threads is
    // alive, and consumers that gave up (a timeout anywhere in the CTA) exit without
    // waiting for their stages; in a normal launch the consumers wait for the same
    // phases, so this wait costs nothing.  It waits for the last kItemSlots items'
    // query rows before the marker is published (the marker completes one more phase
    // of an item slot) and for the last kStages stages after it, each with the full
    // bound kWaitTimeoutNs: neither the launch's wait limit nor the abort flag cuts
    // it short.
    __device__ void finish()
    {
#ifdef PA_TRACE
        if (lane == 0) {
            PA_TRACE_SET(3, dev::global_timer_ns());
            PA_TRACE_SET(4, n);
        }
#endif
        if (lane != 0)
            return;
        for (uint32_t k = n > kItemSlots ? n - kItemSlots : 0; k < n; ++k)
            dev::mbar_wait(dev::smem_addr(&c.item_full[k % kItemSlots]), (k / kItemSlots) & 1u,
                           kWaitTimeoutNs);
        if (!failed) {
            const uint32_t slot = n % kItemSlots;
            if (wait_slot(&c.item_empty[slot], ((n / kItemSlots) & 1u) ^ 1u)) {
                c.items[slot].seq = -1;
                dev::mbar_arrive(dev::smem_addr(&c.item_full[slot]));
            } else {
                failed = true;
            }
        }
        for (uint32_t q = g > kStages ? g - kStages : 0; q < g; ++q)
            dev::mbar_wait(dev::smem_addr(&c.full[q % kStages]), (q / kStages) & 1u,
                           kWaitTimeoutNs);
    }
};

// ---------------------------------------------------------------------------
// Balanced split helpers.  Work is measured in ring stages: a unit of a sequence
// with nb blocks costs kUnitCost + ceil(nb / bps) positions -- the fixed cost of an
// item (descriptor, query rows, block-table lookup latency, merge) counted as
// kUnitCost stages, then its real stages.  All units of all sequences, in order
// (sequence, kv head, head group) -- for the own blocks of a batch with shared
// prefixes, (kv head, head group, sequence) -- form one stream of `total`
// positions; CTA c of G takes positions [c * total / G, (c + 1) * total / G).
// ---------------------------------------------------------------------------
// The units a sequence contributes to the stream of the current pass.
//   pass 0: (kv head, head group) units over blocks [start, nb) -- start is the
//           shared prefix length of a grouped sequence (its rows then merge with the
//           prefix pass's), else 0;
//   pass 1: only the first member of a group has units: (kv head, member group)
//           over the group's shared blocks [0, nb = prefix), each unit holding the
//           query rows of up to 16 / G member sequences.
struct SeqUnits {
    int nunits;   // units of this sequence in the stream
    int ns;       // ring stages per unit
    int start;    // first block
    int nb;       // end block
    int len;      // context length the unit's blocks belong to
    int members;  // pass 1: group size
    int mgroups;  // pass 1: member groups per kv head
};

template <bool kShare>
__device__ __forceinline__ SeqUnits seq_units(const DecodeParams &p, int s, int bs, int bps)
{
    // Every entry of the sequence the walk may need is loaded before any is tested,
    // so that the loads are in flight together: one memory round trip per batch of
    // sequences rather than one per test (length, group, prefix length, members).
    const bool grouped = kShare && p.share != nullptr && p.group <= kHeadsPerItem;
    const bool members = grouped && p.pass == 1;
    const int t = p.context_lens[s];
    const int lead = grouped ? p.share[2 * s] : -1;
    const int sp = grouped ? p.share[2 * s + 1] : 0;
    int v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        v[k] = (members && s + 1 + k < p.num_seqs) ? p.share[2 * (s + 1 + k)] : -1;
    const int cap = p.max_blocks * bs;
    const int len = t < 0 ? 0 : (t > cap ? cap : t);
    // leading blocks shared with the group (0: not grouped)
    const int shared = (lead >= 0 && sp > 0) ? min(sp, p.max_blocks) : 0;

    SeqUnits u;
    u.members = 1;
    u.mgroups = 1;
    if (kShare && p.pass == 1) {
        u.nunits = 0;
        u.ns = 0;
        u.start = 0;
        u.nb = 0;
        u.len = 0;
        if (lead == s && shared > 0) {
            // members follow their first member; past the first eight, eight more
            // entries at a time
            int k = 0;
            while (k < 8 && v[k] == s)
                ++k;
            int m = 1 + k;
            while (k == 8) {
                int w[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    w[j] = (s + m + j < p.num_seqs) ? p.share[2 * (s + m + j)] : -1;
                k = 0;
                while (k < 8 && w[k] == s)
                    ++k;
                m += k;
            }
            const int mpi = members_per_item(p.group);
            u.members = m;
            u.mgroups = (m + mpi - 1) / mpi;
            u.nunits = p.num_kv_heads * u.mgroups;
            u.ns = (shared + bps - 1) / bps;
            u.nb = shared;
            u.len = shared * bs;
        }
        return u;
    }
    const int nb = (len + bs - 1) / bs;
    int P = min(shared, nb);
    if (kShare && P > 0 && len <= shared * bs) {
        // the context ends inside the group's shared blocks (its newest token would
        // sit in a shared block, which the allocator copies on write): an input
        // error, reported; the sequence's own launch reads all its blocks itself and
        // ignores the prefix rows the shared launch computes for it
        atomicOr(p.errors, PA_DEVERR_SHARE);
        P = 0;
    }
    u.nunits = p.num_kv_heads * p.head_groups;
    u.ns = (nb - P + bps - 1) / bps;
    u.start = P;
    u.nb = nb;
    u.len = len;
    return u;
}

// Units of a sequence of the plain decode from its (clamped) context length.
__device__ __forceinline__ SeqUnits seq_units_of_len(const DecodeParams &p, int len, int bs, int bps)
{
    SeqUnits u;
    u.members = 1;
    u.mgroups = 1;
    const int nb = (len + bs - 1) / bs;
    u.nunits = p.num_kv_heads * p.head_groups;
    u.ns = (nb + bps - 1) / bps;
    u.start = 0;
    u.nb = nb;
    u.len = len;
    return u;
}

__device__ __forceinline__ long long warp_sum_ll(long long v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Positions of the whole stream (every lane gets the value).  With kPrefix,
// *prefix tells whether some sequence's units start after shared leading blocks
// (the own blocks of a batch with shared prefixes).
template <bool kShare, bool kPrefix>
__device__ __forceinline__ long long stream_total(const DecodeParams &p, int bs, int bps, int lane,
                                                  long long *units = nullptr,
                                                  bool *prefix = nullptr)
{
    long long t = 0, n = 0;
    bool pre = false;
    for (int s0 = 0; s0 < p.num_seqs; s0 += 32) {
        const int s = s0 + lane;
        if (s < p.num_seqs) {
            const SeqUnits u = seq_units<kShare>(p, s, bs, bps);
            t += (long long)u.nunits * (kUnitCost + u.ns);
            n += u.nunits;
            if (kPrefix)
                pre |= u.start > 0;
        }
    }
    if (units)
        *units = warp_sum_ll(n);
    if (kPrefix)
        *prefix = __any_sync(0xffffffffu, pre);
    return warp_sum_ll(t);
}

// The sequence whose positions contain x (sequences without units have none);
// num_seqs if x >= total.  *base_out gets the sequence's first position.  With
// one_unit, each sequence counts the positions of one of its units (a row of the
// (unit, sequence) order).  Warp-cooperative.
template <bool kShare>
__device__ __forceinline__ int find_seq_at(const DecodeParams &p, int bs, int bps, long long x,
                                           long long *base_out, int lane, bool one_unit = false)
{
    long long base = 0;
    for (int s0 = 0; s0 < p.num_seqs; s0 += 32) {
        const int s = s0 + lane;
        long long w = 0;
        if (s < p.num_seqs) {
            const SeqUnits u = seq_units<kShare>(p, s, bs, bps);
            w = (one_unit ? 1ll : (long long)u.nunits) * (kUnitCost + u.ns);
        }
        long long incl = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o)
                incl += v;
        }
        const long long excl = incl - w;
        const unsigned hit = __ballot_sync(0xffffffffu, s < p.num_seqs && base + incl > x);
        if (hit) {
            const int L = __ffs(hit) - 1;
            *base_out = base + __shfl_sync(0xffffffffu, excl, L);
            return s0 + L;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
    }
    *base_out = base;
    return p.num_seqs;
}

// CTAs the balanced split spreads a stream of `total` positions over: the whole
// grid once each CTA gets at least kMinPositions positions, fewer for small
// batches, where cutting a unit between CTAs costs more (a partial store, a count
// and a merge on the critical path) than the stages it spreads.  The rest of the
// grid exits at once.  (Cutting the stream into more, dynamically claimed chunks
// than CTAs evens out the end of a launch but costs more than it saves here: each
// extra cut adds a split unit, with its fences and count, and a claim round trip.)
// (kMinPositions, balanced_divisor: pa_internal.h.)
__device__ __forceinline__ long long balanced_grid(long long total, int divisor)
{
    return balanced_grid_of(total, divisor, (long long)gridDim.x);
}

// CTA of a G-CTA grid whose stage range contains stream stage x.
__device__ __forceinline__ long long cta_of(long long x, long long total, long long G)
{
    return ((x + 1) * G - 1) / total;
}

// Emits unit u of sequence s (stream positions [a, a + kUnitCost + ns)) if its
// real stages meet the CTA's range [s_c, e_c).  Returns false once the producer
// aborted.
template <bool kShare, class Prod>
__device__ __forceinline__ bool emit_unit(const DecodeParams &p, Prod &pr, const SeqUnits &su,
                                          int s, long long u, long long a, long long s_c,
                                          long long e_c, long long total, long long G,
                                          long long cta, int bps, int div)
{
    const long long ns = su.ns;
    const long long ra = a + kUnitCost;  // first real stage
    const long long rb = ra + ns;
    Item it;
    it.len = su.len;
    it.total_lo = (unsigned int)(total & 0xffffffffll);
    it.total_hi = (unsigned int)(total >> 32);
    it.tseq = s;
    if (kShare && p.pass == 1) {
        const int mpi = members_per_item(p.group);
        const int mg = (int)(u % su.mgroups);
        const int members = min(mpi, su.members - mg * mpi);
        it.seq = s + mg * mpi;
        it.kvh = (int)(u / su.mgroups);
        it.hg = 0;
        it.qrow0 = it.kvh * p.group;
        it.rows = members * p.group;
        it.packed = pack_rows(members, p.group, kToPrefix);
    } else {
        it.seq = s;
        it.kvh = (int)(u / p.head_groups);
        it.hg = (int)(u % p.head_groups);
        it.qrow0 = it.kvh * p.group + it.hg * kHeadsPerItem;
        it.rows = min(kHeadsPerItem, p.group - it.hg * kHeadsPerItem);
        it.packed = pack_rows(1, it.rows, kShare && su.start > 0 ? kMergePrefix : 0);
    }
    it.c_first = -1;
    it.nparts = 0;
    if (ns == 0) {
        // an empty unit belongs to the CTA holding its start: zero rows (or the
        // shared-prefix rows alone)
        if (a < s_c)
            return true;
        it.j0 = it.j1 = su.start;
        it.partial = 0;
        it.prow0 = 0;
    } else {
        const long long lo = max(ra, s_c), hi = min(rb, e_c);
        if (lo >= hi)
            return true;
        it.j0 = su.start + (int)((lo - ra) * bps);
        it.j1 = (int)min(su.start + (hi - ra) * bps, (long long)su.nb);
        it.partial = (lo == ra && hi == rb) ? 0 : 1;
        // slot 2c: the unit's stages began in an earlier CTA; 2c + 1: they go on
        it.prow0 = (int)((2 * cta + (ra < s_c ? 0 : 1)) * kHeadsPerItem);
        if (it.partial) {
            const long long cf = cta_of(ra, total, G);
            const long long cl = cta_of(rb - 1, total, G);
            int np = 1;
            for (long long cc = cf + 1; cc <= cl; ++cc)
                np += (cc * total / G < (cc + 1) * total / G) ? 1 : 0;
            it.c_first = (int)cf;
            it.nparts = np;
        }
    }
    // consecutive items of a CTA start their warp rotation where the stream is
    it.packed = (it.packed & ~(0x3f << 2)) | ((int)((ns == 0 ? a : max(ra, s_c)) & 3) << 2) |
                (div << 4);
    return pr.emit(it);
}

// Stream order (sequence, unit): every unit of a sequence, then the next sequence.
template <bool kShare, class Prod>
__device__ __forceinline__ bool walk_chunk(const DecodeParams &p, int bs, int bps, Prod &pr,
                                           int lane, long long total, long long G, long long cta,
                                           int div)
{
    const long long s_c = cta * total / G;
    const long long e_c = (cta + 1) * total / G;
    if (s_c >= e_c)
        return true;
    long long base = 0;
    int s = find_seq_at<kShare>(p, bs, bps, s_c, &base, lane);
    for (; s < p.num_seqs && base < e_c && !*pr.c.abort; ++s) {
        const SeqUnits su = seq_units<kShare>(p, s, bs, bps);
        if (su.nunits == 0)
            continue;
        const long long span = kUnitCost + su.ns;
        const long long u_lo = s_c > base ? (s_c - base) / span : 0;
        const long long u_hi = min((long long)su.nunits - 1, (e_c - 1 - base) / span);
        for (long long u = u_lo; u <= u_hi; ++u)
            if (!emit_unit<kShare>(p, pr, su, s, u, base + u * span, s_c, e_c, total, G, cta, bps,
                                   div))
                return false;
        base += (long long)su.nunits * span;
    }
    return !*pr.c.abort;
}

// Stream order (unit, sequence), for the own blocks of a batch with shared
// prefixes (pass 0: every sequence has the same units): unit 0 of every sequence,
// then unit 1 of every sequence, ...  A CTA's range then holds one unit of many
// sequences, a mix of own-part lengths, instead of every unit of one or two
// sequences: the per-unit charge misjudges short and long units in opposite
// directions, and a mix averages that out where a run of alike units adds it up.
template <class Prod>
__device__ __forceinline__ bool walk_chunk_unit_major(const DecodeParams &p, int bs, int bps,
                                                      Prod &pr, int lane, long long total,
                                                      long long G, long long cta, int div)
{
    const long long s_c = cta * total / G;
    const long long e_c = (cta + 1) * total / G;
    if (s_c >= e_c)
        return true;
    const long long U = (long long)p.num_kv_heads * p.head_groups;
    const long long W = total / U;  // positions of one unit of every sequence
    long long u = s_c / W;
    long long inner = 0;
    int s = find_seq_at<true>(p, bs, bps, s_c - u * W, &inner, lane, true);
    long long base = u * W + inner;
    for (; u < U && base < e_c && !*pr.c.abort; ++u, s = 0) {
        for (; s < p.num_seqs && base < e_c; ++s) {
            const SeqUnits su = seq_units<true>(p, s, bs, bps);
            if (!emit_unit<true>(p, pr, su, s, u, base, s_c, e_c, total, G, cta, bps, div))
                return false;
            base += kUnitCost + su.ns;
        }
    }
    return !*pr.c.abort;
}

// pa_decode_planned / pa_decode_shared_planned: the walk of the balanced split
// from the CTA's start as the host computed it (pa_decode_plan,
// pa_decode_shared_plan).  The stream total, the CTA's range, its first sequence
// with that sequence's first position and units, and the block ids of its first
// item's first window come from the plan, so the first copies need no pass over
// the context lengths (or the shared-prefix entries) and no block-table read.
// Later sequences' entries are read as the walk reaches them.  The items are the
// ones the walk from scratch emits.  A plan made for other inputs gives wrong rows
// but never an access outside the arguments: every field is bounded before use,
// the CTA count is recomputed from the total as the merge recomputes it, and a
// walk whose positions would pass the total stops and raises PA_DEVERR_PLAN.
template <int kMode, class Prod>
__device__ __forceinline__ void walk_planned(const DecodeParams &p, int bs, int bps, Prod &pr,
                                             int lane)
{
    constexpr bool kShare = kMode == kModePrefix || kMode == kModeOwn;
    const int v = p.plan[(size_t)blockIdx.x * kPlanInts + lane];
    auto get = [&](int f) { return __shfl_sync(0xffffffffu, v, f); };
    auto get64 = [&](int f) {
        return (long long)(unsigned)get(f) | ((long long)get(f + 1) << 32);
    };
    const long long total = max(get64(kPlanTotal), 1ll);
    const int div = min(max(get(kPlanDiv), (int)kMinPositions), 8);
    const long long G = balanced_grid(total, div);
    const int seq = get(kPlanSeq);
    if ((long long)blockIdx.x >= G || seq < 0 || seq >= p.num_seqs)
        return;
    const long long e_c = min(max(get64(kPlanEnd), 0ll), total);
    const long long s_c = min(max(get64(kPlanStart), 0ll), e_c);
    long long base = min(max(get64(kPlanBase), 0ll), s_c);
    const int aux = kShare ? get(kPlanAux) : 0;
    pr.plan_blk = v;
    pr.plan_seq = seq;
    pr.plan_j0 = get(kPlanJ0);
    // the first sequence's units
    SeqUnits su0;
    if constexpr (kMode == kModePrefix) {
        // the group's shared blocks, streamed with the rows of its members
        const int members = min(max(aux & kAuxValueMask, 1), p.num_seqs - seq);
        const int shared = min(max(get(kPlanLen), 0), p.max_blocks);
        const int mpi = members_per_item(p.group);
        su0.members = members;
        su0.mgroups = (members + mpi - 1) / mpi;
        su0.nunits = p.num_kv_heads * su0.mgroups;
        su0.ns = (shared + bps - 1) / bps;
        su0.start = 0;
        su0.nb = shared;
        su0.len = shared * bs;
    } else {
        su0 = seq_units_of_len(p, min(max(get(kPlanLen), 0), p.max_blocks * bs), bs, bps);
        if (kMode == kModeOwn) {
            // its own blocks, after the group's shared ones
            su0.start = min(aux & kAuxValueMask, su0.nb);
            su0.ns = (su0.nb - su0.start + bps - 1) / bps;
            if ((aux & kAuxShareErr) && lane == 0)
                atomicOr(p.errors, PA_DEVERR_SHARE);
        }
    }
    const long long cta = blockIdx.x;
    if (kMode == kModeOwn && (aux & kAuxUnitMajor)) {
        // (unit, sequence) order, as walk_chunk_unit_major
        const long long U = (long long)p.num_kv_heads * p.head_groups;
        const long long W = total / U;
        if (W <= 0)
            return;
        bool first = true;
        int s = seq;
        for (long long u = s_c / W; u < U && base < e_c && !*pr.c.abort; ++u, s = 0) {
            for (; s < p.num_seqs && base < e_c; ++s) {
                const SeqUnits su = first ? su0 : seq_units<true>(p, s, bs, bps);
                first = false;
                if (base + kUnitCost + su.ns > total) {
                    if (lane == 0)
                        atomicOr(p.errors, PA_DEVERR_PLAN);
                    return;
                }
                if (!emit_unit<true>(p, pr, su, s, u, base, s_c, e_c, total, G, cta, bps, div))
                    return;
                base += kUnitCost + su.ns;
            }
        }
        return;
    }
    for (int s = seq; s < p.num_seqs && base < e_c && !*pr.c.abort; ++s) {
        const SeqUnits su = s == seq ? su0 : seq_units<kShare>(p, s, bs, bps);
        if (kShare && su.nunits == 0)
            continue;
        const long long span = kUnitCost + su.ns;
        if (base + (long long)su.nunits * span > total) {
            if (lane == 0)
                atomicOr(p.errors, PA_DEVERR_PLAN);
            return;
        }
        const long long u_lo = s_c > base ? (s_c - base) / span : 0;
        const long long u_hi = min((long long)su.nunits - 1, (e_c - 1 - base) / span);
        for (long long u = u_lo; u <= u_hi; ++u)
            if (!emit_unit<kShare>(p, pr, su, s, u, base + u * span, s_c, e_c, total, G, cta, bps,
                                   div))
                return;
        base += (long long)su.nunits * span;
    }
}

// The producer's walk of the balanced split: CTA c streams positions
// [c * total / G, (c + 1) * total / G).  The own-block launch of the shared-prefix
// decode takes the (unit, sequence) order when the batch has shared prefixes.
template <int kMode, class Prod>
__device__ __forceinline__ void walk_balanced(const DecodeParams &p, int bs, int bps, Prod &pr,
                                              int lane)
{
    constexpr bool kShare = kMode == kModePrefix || kMode == kModeOwn;
    constexpr bool kOwn = kMode == kModeOwn;
    long long units = 0;
    bool prefix = false;
    const long long total = stream_total<kShare, kOwn>(p, bs, bps, lane, &units, &prefix);
    const int div = balanced_divisor(total, units);
    const long long G = balanced_grid(total, div);
    if ((long long)blockIdx.x >= G)
        return;
    if (kOwn && prefix)
        walk_chunk_unit_major(p, bs, bps, pr, lane, total, G, (long long)blockIdx.x, div);
    else
        walk_chunk<kShare>(p, bs, bps, pr, lane, total, G, (long long)blockIdx.x, div);
}

template <class Prod>
__device__ __forceinline__ void walk_fixed(const DecodeParams &p, int bs, Prod &pr, int lane)
{
    int seq = 0;
    long long base = 0;
    for (long long w = blockIdx.x;; w += gridDim.x) {
        if (!find_item(p, bs, w, seq, base, lane) || *pr.c.abort)
            break;
        if (!pr.emit(decode_item(p, bs, w, seq, base)))
            return;
    }
}

template <typename T, int D, int BS, int kBPS, int kChunks, int kTileBytes, int kStages,
          int kMode, int kCopy>
__device__ __forceinline__ void producer_loop(const DecodeParams &p, const CUtensorMap *tk,
                                              const CUtensorMap *tv, const CtaState &c, int lane)
{
    Producer<T, D, BS, kBPS, kChunks, kTileBytes, kStages, kCopy> pr(p, tk, tv, c, lane);
    constexpr bool kShare = kMode == kModePrefix || kMode == kModeOwn;
    if constexpr (kMode == kModePlan)
        walk_planned<kModePlan>(p, BS, kBPS, pr, lane);
    else if (kShare && p.plan != nullptr)
        walk_planned<kMode>(p, BS, kBPS, pr, lane);
    else if (p.balanced)
        walk_balanced<kMode>(p, BS, kBPS, pr, lane);
    else
        walk_fixed(p, BS, pr, lane);
    pr.finish();
}

// ---------------------------------------------------------------------------
// Final value of element `col` of item row r: normalised output o and the row's
// log2-sum-exp.  Goes to the output (cast to T), to the shared-prefix buffer
// (prefix pass), or is first merged with the shared-prefix row by the
// log-sum-exp rule (own blocks of a grouped sequence).
// ---------------------------------------------------------------------------
template <typename T, int D, bool kShare>
__device__ __forceinline__ void store_result(const DecodeParams &p, const Item &it, int r, int col,
                                             float o, float lse, const float *pfx_s)
{
    constexpr int PS = D + kPfxPad;
    const int rpm = it.rpm();
    const size_t row = (size_t)(it.seq + r / rpm) * p.num_q_heads + it.qrow0 + r % rpm;
    const int f = it.flags();
    if (kShare && (f & kToPrefix)) {
        p.pfx[row * PS + col] = o;
        if (col == 0)
            p.pfx[row * PS + D] = lse;
        return;
    }
    if (kShare && (f & kMergePrefix)) {
        // the item's prefix rows, staged in shared memory when the item started
        const float lp = pfx_s[r * PS + D];
        const float m2 = fmaxf(lse, lp);
        if (m2 != -INFINITY) {
            const float wa = exp2f(lse - m2), wb = exp2f(lp - m2);
            o = (wa * o + wb * pfx_s[r * PS + col]) / (wa + wb);
        }
    }
    reinterpret_cast<T *>(p.out)[row * D + col] = dev::from_float<T>(o);
}

// Pass 0 of the shared-prefix decode: start copying the item's prefix rows (o and
// log2-sum-exp, written by pass 1) into buffer `buf` with per-thread asynchronous
// copies; the consumers wait for them (cp.async.wait_all) before the barrier that
// precedes the item's final store.  The two buffers alternate by item, so this
// item's copies never land under a warp still merging the previous item.
template <int D>
__device__ __forceinline__ void stage_prefix(const DecodeParams &p, const Item &it, float *buf,
                                             int tid)
{
    constexpr int PS = D + kPfxPad;
    const float *src = p.pfx + ((size_t)it.seq * p.num_q_heads + it.qrow0) * PS;
    const int units = it.rows * PS / 4;  // 16-byte units
    for (int k = tid; k < units; k += 32 * kConsumerWarps)
        dev::cp_async16(dev::smem_addr(buf + 4 * k), src + 4 * k);
    dev::cp_async_commit();
}

// ---------------------------------------------------------------------------
// Merge the four consumer states of one item and store it.
// ---------------------------------------------------------------------------
template <typename T, int D, bool kShare>
__device__ __forceinline__ void finalize_item(const DecodeParams &p, const Item &it, float *acc,
                                              const float *ml, int rows_cap, int tid,
                                              const float *pfx_s, bool own_in_smem)
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
        if (!it.partial) {
            store_result<T, D, kShare>(p, it, r, col, o, (L > 0.f) ? M + log2f(L) : -INFINITY,
                                       pfx_s);
        } else if (own_in_smem) {
            // this CTA completes the unit now: its rows stay here, in the first warp's
            // accumulator rows (each element read, then written, by this thread alone);
            // the merge recomputes their log2-sum-exp from `ml`
            acc[r * S + col] = o;
        } else {
            const size_t pr = (size_t)it.prow0 + r;
            p.part_o[pr * D + col] = o;
            if (col == 0)
                p.part_lse[pr] = (L > 0.f) ? M + log2f(L) : -INFINITY;
        }
    }
}

// ---------------------------------------------------------------------------
// Balanced split: merge of a unit whose stages several CTAs shared.  Each CTA
// writes its partial (fp32 output rows + log2-sum-exp), releases it with a GPU-scope
// fence and counts it on the unit's counter; the CTA whose count completes the set
// takes an acquire fence and merges every partial with the log-sum-exp rule.  No CTA waits for
// another.  Counters hold (epoch << 32 | count): a value left by an earlier call
// carries another epoch and counts as zero, so they never need clearing.  The CTA
// that completes a unit also resets its counter to zero, so a completed launch leaves
// every counter it used at zero: the replays of a captured CUDA graph reuse one
// epoch, and each starts from clean counters.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool count_partial(const DecodeParams &p, const Item &it,
                                              unsigned long long old)
{
    unsigned long long *ctr = p.counters + it.c_first;
    unsigned int cnt;
    for (;;) {  // each failed exchange means another CTA counted: at most nparts rounds
        cnt = (unsigned int)(old >> 32) == p.epoch ? (unsigned int)old : 0u;
        const unsigned long long want = ((unsigned long long)p.epoch << 32) | (cnt + 1u);
        const unsigned long long prev = atomicCAS(ctr, old, want);
        if (prev == old)
            break;
        old = prev;
    }
    const bool last = cnt + 1u == (unsigned int)it.nparts;
    if (last)  // every part is counted: no other CTA touches this counter again
        *reinterpret_cast<volatile unsigned long long *>(ctr) = 0ull;
    return last;
}

// Before the item's final barrier, thread 0 of a CTA holding one of the two parts of
// a unit cut once reads the unit's counter.  When the other part is counted
// already, this CTA completes the unit: after an acquire fence (the other part's
// rows were released before its count) it merges them with its own rows, kept in
// shared memory, and neither stores, fences nor counts its own (*c.merge = 2).
// Otherwise the count follows the usual release (finish_item), from the value read
// here.  Units cut more than once skip the early read: their parts tend to finish
// together, and a value read early would only make their exchanges fail.
__device__ __forceinline__ void probe_split_last(const DecodeParams &p, const Item &it,
                                                 const CtaState &c)
{
    int early = 0;
    if (p.balanced && it.partial) {
        const unsigned long long v =
            *reinterpret_cast<volatile unsigned long long *>(p.counters + it.c_first);
        *c.ctr_seen = v;
        const unsigned int cnt = (unsigned int)(v >> 32) == p.epoch ? (unsigned int)v : 0u;
        if (it.nparts == 2 && cnt == 1u) {
            dev::fence_acq_rel_gpu();
            early = 1;
            // the other part is counted and this one never will be: reset for the
            // next launch (see count_partial)
            *reinterpret_cast<volatile unsigned long long *>(p.counters + it.c_first) = 0ull;
        }
    }
    *c.merge = early ? 2 : 0;
}

// Log2-sum-exp of row r of this CTA's own part, from the consumer warps' (max, sum).
__device__ __forceinline__ float own_lse(const float *ml, int r)
{
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
    float L = 0.f;
    if (any) {
#pragma unroll
        for (int c = 0; c < kConsumerWarps; ++c) {
            const float mc = ml[(c * kHeadsPerItem + r) * 2];
            if (mc != -INFINITY)
                L += exp2f(mc - M) * ml[(c * kHeadsPerItem + r) * 2 + 1];
        }
    }
    return L > 0.f ? M + log2f(L) : -INFINITY;
}

// Partial row i (0-based) of a split unit: slot 2 c_first + 1, then slot 2 c of the
// next CTAs that hold stages (a CTA range is empty only when the stream has fewer
// positions than the grid has CTAs; otherwise the CTAs are consecutive).
__device__ __forceinline__ long long split_slot(const Item &it, int i, long long total, long long G)
{
    if (i == 0)
        return 2ll * it.c_first + 1;
    if (total >= G)
        return 2ll * (it.c_first + i);
    long long cc = it.c_first;
    for (int k = 0; k < i; ++k)
        do {
            ++cc;
        } while (cc * total / G >= (cc + 1) * total / G);
    return 2 * cc;
}

// Merge the nparts partials of a split unit into its output rows: one warp per
// query head; lane i holds partial i's log2-sum-exp.
// own_o: this CTA's own rows (row stride D + kAccPad) when it completes a unit cut
// once early (probe_split_last), with their log2-sum-exp from own_ml; null when its
// part went through the partial slots.
template <typename T, int D, bool kShare>
__device__ __forceinline__ void merge_split_unit(const DecodeParams &p, const Item &it, int warp,
                                              int lane, const float *pfx_s,
                                              const float *own_o = nullptr,
                                              const float *own_ml = nullptr)
{
    constexpr int VEC = D / 32;
    constexpr int S = D + kAccPad;
    const long long total = ((long long)it.total_hi << 32) | (long long)it.total_lo;
    const long long G = balanced_grid(total, it.divisor());
    for (int r = warp; r < it.rows; r += kConsumerWarps) {
        if (it.nparts == 2) {
            // the usual case (a unit cut once): both parts' loads in flight at once
            const int r0 = (int)split_slot(it, 0, total, G) * kHeadsPerItem + r;
            const int r1 = (int)split_slot(it, 1, total, G) * kHeadsPerItem + r;
            const int own = own_o ? it.prow0 + r : -1;
            const bool o0 = r0 == own, o1 = r1 == own;
            const float lo = own_o ? own_lse(own_ml, r) : 0.f;
            const float l0 = o0 ? lo : __ldcg(p.part_lse + r0);
            const float l1 = o1 ? lo : __ldcg(p.part_lse + r1);
            float v0[VEC], v1[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v0[e] = o0 ? own_o[r * S + lane * VEC + e]
                           : __ldcg(p.part_o + (size_t)r0 * D + lane * VEC + e);
                v1[e] = o1 ? own_o[r * S + lane * VEC + e]
                           : __ldcg(p.part_o + (size_t)r1 * D + lane * VEC + e);
            }
            const float M = fmaxf(l0, l1);
            const float w0 = exp2f(l0 - M), w1 = exp2f(l1 - M);
            const float W = w0 + w1;
            const float lse = M + log2f(W);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                store_result<T, D, kShare>(p, it, r, lane * VEC + e,
                                           (w0 * v0[e] + w1 * v1[e]) / W, lse, pfx_s);
            continue;
        }
        float M = -INFINITY;
        for (int i0 = 0; i0 < it.nparts; i0 += 32) {
            const int i = i0 + lane;
            if (i < it.nparts)
                M = fmaxf(M, __ldcg(p.part_lse + split_slot(it, i, total, G) * kHeadsPerItem + r));
        }
        M = dev::warp_max(M);
        float W = 0.f;
        float acc[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            acc[e] = 0.f;
        for (int i0 = 0; i0 < it.nparts; i0 += 32) {
            const int i = i0 + lane;
            long long row = 0;
            float wgt = 0.f;
            if (i < it.nparts) {
                row = split_slot(it, i, total, G) * kHeadsPerItem + r;
                wgt = exp2f(__ldcg(p.part_lse + row) - M);
            }
            W += wgt;
            const int n = min(32, it.nparts - i0);
            for (int k0 = 0; k0 < n; k0 += 4) {
                float v[4][VEC], wk[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = min(k0 + u, n - 1);
                    const long long rk = __shfl_sync(0xffffffffu, row, k);
                    wk[u] = (k0 + u < n) ? __shfl_sync(0xffffffffu, wgt, k) : 0.f;
                    const float *po = p.part_o + rk * D + lane * VEC;
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        v[u][e] = __ldcg(po + e);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        acc[e] = fmaf(wk[u], v[u][e], acc[e]);
            }
        }
        W = dev::warp_sum(W);
        const float lse = M + log2f(W);
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            store_result<T, D, kShare>(p, it, r, lane * VEC + e, acc[e] / W, lse, pfx_s);
    }
}

// End of an item for the consumer warps: shared-memory reuse barrier and, for a
// split unit of the balanced schedule, the count-and-merge step.  The barrier
// orders every consumer thread's partial stores before thread 0's release fence and
// count (fences are cumulative over what thread 0 has observed); the merging CTA's
// acquire fence, then the next barrier, let all its threads see the other partials.
// False on a timeout.
template <typename T, int D, bool kShare>
__device__ __forceinline__ bool finish_item(const DecodeParams &p, const Item &it, const CtaState &c,
                                            uint32_t &sph, int warp, int lane, const float *pfx_s)
{
    const bool split = p.balanced && it.partial;
    if (!consumer_sync(p, c, sph))
        return false;
    if (!split)
        return true;
    if (*c.merge == 2) {
        // completes the unit (probe_split_last): own rows from shared memory, then a
        // barrier before the next item may overwrite them
        merge_split_unit<T, D, kShare>(p, it, warp, lane, pfx_s, c.macc, c.mml);
        return consumer_sync(p, c, sph);
    }
    if (threadIdx.x == 0) {
        // release: this CTA's partial rows (observed through the barrier above)
        // become visible before the count; acquire, only in the CTA that completes
        // the set: it then sees every other partial and passes that on through the
        // next barrier
        dev::fence_acq_rel_gpu();
        const bool last = count_partial(p, it, *c.ctr_seen);
        if (last)
            dev::fence_acq_rel_gpu();
        *c.merge = last ? 1 : 0;
    }
    if (!consumer_sync(p, c, sph))
        return false;
    if (*c.merge)
        merge_split_unit<T, D, kShare>(p, it, warp, lane, pfx_s);
    return true;
}

// ---------------------------------------------------------------------------
// Fused append: copy the newest token's K and V rows (staged by the producer next
// to the stage) into row `r` of the stage's swizzled tiles, and store them into the
// cache at (physical block, r % block_size).  Nothing else in the launch reads those
// cache bytes: only this (sequence, kv head) unit covers them, and it uses the
// staged copy.  One 16-byte unit per lane per pass.  append_ok false (a planned
// item whose context length is not the one the launch reads): the tile is patched
// but nothing is stored to the cache, and PA_DEVERR_PLAN is raised.
// ---------------------------------------------------------------------------
template <typename T, int D, int BS>
__device__ __forceinline__ void patch_newest_row(const DecodeParams &p, const Item &it,
                                              const CtaState &c, uint32_t st, uint8_t *stage,
                                              int lane, bool append_ok)
{
    using C = Cfg<T, D, BS>;
    constexpr int kUnits = D * (int)sizeof(T) / 16;  // 16-byte units per row
    constexpr int kUnitElems = 16 / (int)sizeof(T);
    constexpr int kCE = 128 / (int)sizeof(T);
    const int r = c.newinfo[2 * st];
    const int blk = c.newinfo[2 * st + 1];
    const uint8_t *staged = c.newrow + (size_t)st * 2 * D * sizeof(T);
    const size_t dst = (((size_t)blk * BS + r % BS) * p.num_kv_heads + it.kvh) * D;
    const bool store = append_ok && it.hg == 0 && blk >= 0 && blk < p.num_blocks;
    if (!append_ok && lane == 0)
        atomicOr(p.errors, PA_DEVERR_PLAN);
    for (int idx = lane; idx < 2 * kUnits; idx += 32) {
        const bool isv = idx >= kUnits;
        const int u = isv ? idx - kUnits : idx;
        const uint4 val = *reinterpret_cast<const uint4 *>(staged + (isv ? D * sizeof(T) : 0) + u * 16);
        const int d0 = u * kUnitElems;
        const int ch = d0 / kCE;
        const int uc = (d0 % kCE) / kUnitElems;
        *reinterpret_cast<uint4 *>(stage + (r / BS) * C::kBlockStride + (isv ? C::kBlockTile : 0) +
                                   ch * (BS * 128) + (r % BS) * 128 + ((uc ^ (r & 7)) << 4)) = val;
        if (store)
            *reinterpret_cast<uint4 *>(reinterpret_cast<T *>(isv ? p.v_cache : p.k_cache) + dst + d0) =
                val;
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// One item of at most 8 query rows on one consumer warp (its share of the
// item's stages), in transposed form: S^T = K Q^T and O^T = V^T P^T.  Tokens
// (scores) and head dims (output) take the MMA's 16-row side, the query rows
// its 8-column side, so a 32-token stage costs 16 + 16 MMAs instead of the
// 32 + 32 that the 16-row form spends on mostly empty rows.  The score
// fragment turns into the B operand of P V by one movmatrix transpose per
// 8 x 8 half.  Ends with the warp's partial rows in its merge area.
// ---------------------------------------------------------------------------
template <typename T, int D, int BS>
__device__ __forceinline__ bool consume_item_n8(const DecodeParams &p, const CtaState &c,
                                                const Item &it, uint32_t slot, uint32_t &g,
                                                int warp, int lane, int rows_cap, bool append_ok)
{
    using C = Cfg<T, D, BS>;
    constexpr int kCE = C::kChunkElems;
    constexpr int TS = C::kStageTokens;  // token rows per stage tile
    constexpr int MT = TS / 16;          // 16-token tiles of S^T (= k-steps of P V)
    constexpr int KS = D / 16;           // k-steps of K Q^T
    constexpr int DM = D / 16;           // 16-dim tiles of O^T
    constexpr int SA = D + kAccPad;
    constexpr uint32_t kQSlotBytes = kHeadsPerItem * D * sizeof(T);
    const int q4 = lane & 3;             // fragment columns: query rows 2 q4, 2 q4 + 1
    const int r8 = lane >> 2;            // fragment row: token (S^T) or dim (O^T)
    const int mi = lane >> 3;            // ldmatrix: which 8x8 matrix this lane addresses
    const int swz = lane & 7;            // 128-byte swizzle: 16-byte unit ^= row % 8
    const bool qlive = r8 < it.rows;

    // Q^T as the B operand (k = head dim, n = query row): plain ldmatrix of the
    // query rows; rows past the item are zero.
    uint32_t qb[KS][2];
    {
        const uint32_t qbase = dev::smem_addr(c.qslots + slot * kQSlotBytes) +
                               (uint32_t)((lane & 7) * D * sizeof(T));
#pragma unroll
        for (int kk = 0; kk < KS / 2; ++kk) {
            uint32_t x0, x1, x2, x3;
            dev::ldsm_x4(qbase + (uint32_t)((kk * 32 + mi * 8) * sizeof(T)), x0, x1, x2, x3);
            qb[2 * kk][0] = qlive ? x0 : 0u;
            qb[2 * kk][1] = qlive ? x1 : 0u;
            qb[2 * kk + 1][0] = qlive ? x2 : 0u;
            qb[2 * kk + 1][1] = qlive ? x3 : 0u;
        }
        uint32_t all = (uint32_t)(it.seq ^ it.kvh ^ it.hg ^ it.len ^ it.j0 ^ it.j1 ^ it.qrow0 ^
                                  it.rows ^ it.partial ^ it.prow0 ^ it.tseq ^ it.packed ^
                                  it.c_first ^ it.nparts) ^
                       it.total_lo ^ it.total_hi;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
            all ^= qb[ks][0] ^ qb[ks][1];
        all = __reduce_xor_sync(0xffffffffu, all);
        if (lane == 0)
            dev::settle_loads(&c.sink[warp], all);
        __syncwarp();
        if (lane == 0)
            dev::mbar_arrive(dev::smem_addr(&c.item_empty[slot]));
    }

    float o[DM][4];
#pragma unroll
    for (int i = 0; i < DM; ++i)
        o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY;  // running max of rows 2 q4 and 2 q4 + 1
    float la = 0.f, lb = 0.f;              // this lane's share of their exp sums
    const int rot = it.rot();
    for (int j = it.j0; j < it.j1; j += C::kBPS, ++g) {
        if (((j - it.j0) / C::kBPS + rot) % kConsumerWarps != warp)
            continue;
        const uint32_t st = g % C::kStages;
#ifdef PA_TRACE
        const unsigned long long t_sw = trace_clock();
#endif
        if (!warp_wait(p, c, &c.full[st], (g / C::kStages) & 1u)) {
            return false;
        }
#ifdef PA_TRACE
        if (threadIdx.x == 0) {
            const unsigned long long t_now = trace_clock();
            PA_TRACE_ADD(13, t_now - t_sw);
            PA_TRACE_SET(11, t_now);
            if (trace_first_tile(p.pass)) {
                PA_TRACE_SET(1, t_now);
            }
        }
#endif
        const int valid = min(min(C::kBPS, it.j1 - j) * BS, it.len - j * BS);
        const uint32_t kb = dev::smem_addr(c.ring + (size_t)st * C::kStageBytes);
        const uint32_t vb = kb + C::kBlockTile;
        if (c.newinfo[2 * st] >= 0)
            patch_newest_row<T, D, BS>(p, it, c, st, c.ring + (size_t)st * C::kStageBytes, lane,
                                       append_ok);

        // S^T = K Q^T: the K tile (rows = tokens) is the row-major A operand.
        // Two accumulators per token tile (even / odd k-steps) shorten the chains.
        const uint32_t krow = kb + (uint32_t)(((mi & 1) * 8 + (lane & 7)) * 128);
        float s[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                s[mt][h][0] = s[mt][h][1] = s[mt][h][2] = s[mt][h][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int d = ks * 16 + (mi >> 1) * 8;
            const uint32_t colpart = (uint32_t)(d / kCE) * (BS * 128) +
                                     (uint32_t)((((d % kCE) >> 3) ^ swz) << 4);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                uint32_t a[4];
                const int tok = mt * 16 + (mi & 1) * 8 + (lane & 7);
                if constexpr (C::kBPS == 1)
                    dev::ldsm_x4(kb + colpart + tok * 128, a[0], a[1], a[2], a[3]);
                else
                    dev::ldsm_x4(krow + colpart + tile_at<BS, C::kBlockStride>(mt * 16), a[0],
                                 a[1], a[2], a[3]);
                dev::Mma<T>::run(s[mt][ks & 1], a, qb[ks][0], qb[ks][1]);
            }
        }

        // scores of tokens mt*16 + r8 (+8) for rows 2 q4, 2 q4 + 1: mask, scale, max
        float mxa = -INFINITY, mxb = -INFINITY;
        float sc[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sc[mt][e] = s[mt][0][e] + s[mt][1][e];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const bool ok = mt * 16 + r8 + 8 * h < valid;
                sc[mt][2 * h] = ok ? sc[mt][2 * h] * p.scale_log2 : -INFINITY;
                sc[mt][2 * h + 1] = ok ? sc[mt][2 * h + 1] * p.scale_log2 : -INFINITY;
                mxa = fmaxf(mxa, sc[mt][2 * h]);
                mxb = fmaxf(mxb, sc[mt][2 * h + 1]);
            }
        }
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) {
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, o_));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, o_));
        }
        const float na = fmaxf(ma, mxa), nb = fmaxf(mb, mxb);
        const float ca = exp2f(ma - na), cb = exp2f(mb - nb);
        ma = na;
        mb = nb;
        float pa = 0.f, pb = 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                sc[mt][2 * h] = exp2f(sc[mt][2 * h] - na);
                sc[mt][2 * h + 1] = exp2f(sc[mt][2 * h + 1] - nb);
                pa += sc[mt][2 * h];
                pb += sc[mt][2 * h + 1];
            }
        }
        la = la * ca + pa;
        lb = lb * cb + pb;
        if (__any_sync(0xffffffffu, ca != 1.f || cb != 1.f)) {
#pragma unroll
            for (int i = 0; i < DM; ++i) {
                o[i][0] *= ca;
                o[i][1] *= cb;
                o[i][2] *= ca;
                o[i][3] *= cb;
            }
        }

        // O^T += V^T P^T: ldmatrix.trans of the V tile (rows = tokens) gives the
        // row-major A operand (m = head dim, k = token); P^T is the B operand.
        const bool partial = valid < TS;
        const uint32_t vrow = vb + (uint32_t)(((mi >> 1) * 8 + (lane & 7)) * 128);
#pragma unroll
        for (int kt = 0; kt < MT; ++kt) {
            const uint32_t pb0 = dev::movmatrix_trans(dev::Mma<T>::pack(sc[kt][0], sc[kt][1]));
            const uint32_t pb1 = dev::movmatrix_trans(dev::Mma<T>::pack(sc[kt][2], sc[kt][3]));
            // stale rows past the context may hold anything (NaN): zero them
            uint32_t mk0 = 0xffffffffu, mk1 = 0xffffffffu;
            if (partial) {
                const int t0 = kt * 16 + 2 * q4;
                mk0 = (t0 < valid ? 0x0000ffffu : 0u) | (t0 + 1 < valid ? 0xffff0000u : 0u);
                mk1 = (t0 + 8 < valid ? 0x0000ffffu : 0u) | (t0 + 9 < valid ? 0xffff0000u : 0u);
            }
#pragma unroll
            for (int dm = 0; dm < DM; ++dm) {
                const int d = dm * 16 + (mi & 1) * 8;
                const int tok = kt * 16 + (mi >> 1) * 8 + (lane & 7);
                const uint32_t addr =
                    C::kBPS == 1 ? vb + (uint32_t)(d / kCE) * (TS * 128) + tok * 128 +
                                       (uint32_t)((((d % kCE) >> 3) ^ swz) << 4)
                                 : vrow + tile_at<BS, C::kBlockStride>(kt * 16) +
                                       (uint32_t)(d / kCE) * (BS * 128) +
                                       (uint32_t)((((d % kCE) >> 3) ^ swz) << 4);
                uint32_t a[4];
                dev::ldsm_x4_trans(addr, a[0], a[1], a[2], a[3]);
                a[0] &= mk0;
                a[1] &= mk0;
                a[2] &= mk1;
                a[3] &= mk1;
                dev::Mma<T>::run(o[dm], a, pb0, pb1);
            }
        }
        __syncwarp();
        if (lane == 0)
            dev::mbar_arrive(dev::smem_addr(&c.empty[st]));
    }

    // partial rows of this warp: O^T fragment (dim dm*16 + r8 (+8), rows 2 q4, 2 q4 + 1)
#pragma unroll
    for (int o_ = 4; o_ < 32; o_ <<= 1) {
        la += __shfl_xor_sync(0xffffffffu, la, o_);
        lb += __shfl_xor_sync(0xffffffffu, lb, o_);
    }
    float *mine = c.macc + warp * rows_cap * SA;
    const int ra = 2 * q4, rb = 2 * q4 + 1;
    if (ra < it.rows) {
#pragma unroll
        for (int dm = 0; dm < DM; ++dm) {
            mine[ra * SA + dm * 16 + r8] = o[dm][0];
            mine[ra * SA + dm * 16 + r8 + 8] = o[dm][2];
        }
    }
    if (rb < it.rows) {
#pragma unroll
        for (int dm = 0; dm < DM; ++dm) {
            mine[rb * SA + dm * 16 + r8] = o[dm][1];
            mine[rb * SA + dm * 16 + r8 + 8] = o[dm][3];
        }
    }
    if (r8 == 0) {
        c.mml[(warp * kHeadsPerItem + ra) * 2] = (ra < it.rows && la > 0.f) ? ma : -INFINITY;
        c.mml[(warp * kHeadsPerItem + ra) * 2 + 1] = la;
        c.mml[(warp * kHeadsPerItem + rb) * 2] = (rb < it.rows && lb > 0.f) ? mb : -INFINITY;
        c.mml[(warp * kHeadsPerItem + rb) * 2 + 1] = lb;
    }
    return true;
}

// ---------------------------------------------------------------------------
// fp16 / bf16 partition kernel: tensor-core consumers.  kMode: the launch it is
// built for (kModePlain, kModePlan, kModePrefix, kModeOwn); kCopy: kCopyJoint or
// kCopySplit, by the caches' placement.
// ---------------------------------------------------------------------------
template <typename T, int D, int BS, bool N8, int kMode, int kCopy>
__global__ void __launch_bounds__(kThreads, 2)
    pa_decode_mma_kernel(const __grid_constant__ DecodeParams p,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v)
{
    using C = Cfg<T, D, BS>;
    constexpr int kCE = C::kChunkElems;
    constexpr int TS = C::kStageTokens;  // token rows per stage tile
    constexpr int NT = TS / 8;   // score n-tiles of 8 tokens
    constexpr int KS = D / 16;   // k-steps of Q K^T
    constexpr int DT = D / 8;    // output n-tiles of 8 dims
    constexpr int SA = D + kAccPad;
    constexpr uint32_t kQSlotBytes = kHeadsPerItem * D * sizeof(T);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int rows_cap = item_rows_cap(p);
    constexpr bool kShare = kMode == kModePrefix || kMode == kModeOwn;
    const int pfx_rows = kShare ? item_pfx_rows(p) : 0;
    const SmemLayout lay =
        make_layout(C::kStages, C::kStageBytes, rows_cap, D, sizeof(T), pfx_rows);
    const CtaState c = cta_state(smem, lay, C::kStages);
    init_cta(p, c, C::kStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (warp == kConsumerWarps) {
        producer_loop<T, D, BS, C::kBPS, C::kChunks, C::kTileBytes, C::kStages, kMode, kCopy>(
            p, &tmap_k, &tmap_v, c, lane);
        return;
    }

    // ---- consumers ----
    const int r0 = lane >> 2;        // fragment row (query head) and row + 8
    const int cq = (lane & 3) * 2;   // fragment column pair
    const int mi = lane >> 3;        // ldmatrix: which 8x8 matrix this lane addresses
    const int swz = lane & 7;        // 128-byte swizzle: 16-byte unit ^= row % 8
    uint32_t g = 0;                  // stages consumed (same count in every warp)
    uint32_t sph = 0;                // consumer barrier phase
#ifdef PA_TRACE
    if (threadIdx.x == 0) {
        unsigned int smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        PA_TRACE_SET(0, dev::global_timer_ns());
        PA_TRACE_SET(8, smid);
    }
    bool first_tile = true;
#endif
    bool pfx_ready = !kShare || !defers_dependency(p);  // prefix rows may be read
    for (uint32_t n = 0;; ++n) {
        const uint32_t slot = n % kItemSlots;
#ifdef PA_TRACE
        const unsigned long long t_iw = trace_clock();
#endif
        if (!warp_wait(p, c, &c.item_full[slot], (n / kItemSlots) & 1u)) {
            break;
        }
#ifdef PA_TRACE
        if (threadIdx.x == 0)
            PA_TRACE_ADD(12, trace_clock() - t_iw);
#endif
        const Item it = load_item(&c.items[slot]);
        if (it.seq < 0)
            break;
        // a planned first item takes its length from the plan: its append is stored
        // only if that is the length the launch reads (read here, used stages later)
        const bool append_ok = (kMode != kModePlan && (kMode != kModeOwn || p.plan == nullptr)) ||
                               p.k_new == nullptr || clamp_len(p, it.tseq, BS) == it.len;
        const bool merge_pfx = kShare && (it.flags() & kMergePrefix) != 0;
        float *pfx_s = c.pfx + (n & 1) * pfx_rows * (D + kPfxPad);
        if (merge_pfx && pfx_ready)
            stage_prefix<D>(p, it, pfx_s, threadIdx.x);
        if constexpr (N8) {
            if (!consume_item_n8<T, D, BS>(p, c, it, slot, g, warp, lane, rows_cap, append_ok))
                break;
        } else {
        const bool live0 = r0 < it.rows, live1 = r0 + 8 < it.rows;

        // Query fragments (A operand of Q K^T) from the item slot; rows past the
        // group are zero.
        uint32_t qa[KS][4];
        {
            const uint32_t qb = dev::smem_addr(c.qslots + slot * kQSlotBytes) +
                                (uint32_t)(((mi & 1) * 8 + (lane & 7)) * D * sizeof(T));
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                dev::ldsm_x4(qb + (uint32_t)((ks * 16 + (mi >> 1) * 8) * sizeof(T)), qa[ks][0],
                             qa[ks][1], qa[ks][2], qa[ks][3]);
                qa[ks][0] = live0 ? qa[ks][0] : 0u;
                qa[ks][2] = live0 ? qa[ks][2] : 0u;
                qa[ks][1] = live1 ? qa[ks][1] : 0u;
                qa[ks][3] = live1 ? qa[ks][3] : 0u;
            }
            // every read of the slot (query rows, descriptor) must have completed
            // before the slot is handed back to the producer
            uint32_t all = (uint32_t)(it.seq ^ it.kvh ^ it.hg ^ it.len ^ it.j0 ^ it.j1 ^ it.qrow0 ^
                                      it.rows ^ it.partial ^ it.prow0 ^ it.tseq ^ it.packed ^
                                      it.c_first ^ it.nparts) ^
                           it.total_lo ^ it.total_hi;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
                all ^= qa[ks][0] ^ qa[ks][1] ^ qa[ks][2] ^ qa[ks][3];
            all = __reduce_xor_sync(0xffffffffu, all);
            if (lane == 0)
                dev::settle_loads(&c.sink[warp], all);
            __syncwarp();
            if (lane == 0)
                dev::mbar_arrive(dev::smem_addr(&c.item_empty[slot]));
        }

        float acc[DT][4];
#pragma unroll
        for (int i = 0; i < DT; ++i)
            acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        float mrow0 = -INFINITY, mrow1 = -INFINITY, lrow0 = 0.f, lrow1 = 0.f;
        bool alive = true;

        const int rot = it.rot();
        for (int j = it.j0; j < it.j1; j += C::kBPS, ++g) {
            if (((j - it.j0) / C::kBPS + rot) % kConsumerWarps != warp)
                continue;
            const uint32_t st = g % C::kStages;
#ifdef PA_TRACE
            const unsigned long long t_sw = trace_clock();
#endif
            if (!warp_wait(p, c, &c.full[st], (g / C::kStages) & 1u)) {
                alive = false;
                break;
            }
#ifdef PA_TRACE
            if (threadIdx.x == 0) {
                const unsigned long long t_now = trace_clock();
                PA_TRACE_ADD(13, t_now - t_sw);
                PA_TRACE_SET(11, t_now);
                if (first_tile) {
                    PA_TRACE_SET(1, t_now);
                    first_tile = false;
                }
            }
#endif
            // tokens of this stage that count: the loaded blocks, up to the context
            const int valid = min(min(C::kBPS, it.j1 - j) * BS, it.len - j * BS);
            const uint32_t kb = dev::smem_addr(c.ring + (size_t)st * C::kStageBytes);
            const uint32_t vb = kb + C::kBlockTile;
            if (c.newinfo[2 * st] >= 0)
                patch_newest_row<T, D, BS>(p, it, c, st, c.ring + (size_t)st * C::kStageBytes, lane,
                                           append_ok);

            // S = Q K^T: K tile rows are tokens, so plain ldmatrix yields the
            // "col" B fragment (k = head dim, n = token).
            const uint32_t krow = kb + (uint32_t)(((mi >> 1) * 8 + (lane & 7)) * 128);
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
                    uint32_t b0, b1, b2, b3;
                    dev::ldsm_x4(krow + colpart + tile_at<BS, C::kBlockStride>(np * 16), b0, b1,
                                 b2, b3);
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
            const bool partial = valid < TS;
            const uint32_t vrow = vb + (uint32_t)(((mi & 1) * 8 + (lane & 7)) * 128);
#pragma unroll
            for (int kt = 0; kt < TS / 16; ++kt) {
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
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    const int d = dp * 16 + (mi >> 1) * 8;
                    const uint32_t addr = vrow + tile_at<BS, C::kBlockStride>(kt * 16) +
                                          (uint32_t)(d / kCE) * (BS * 128) +
                                          (uint32_t)((((d % kCE) >> 3) ^ swz) << 4);
                    uint32_t v0, v1, v2, v3;
                    dev::ldsm_x4_trans(addr, v0, v1, v2, v3);
                    dev::Mma<T>::run(acc[2 * dp], pa, v0 & mk0, v1 & mk1);
                    dev::Mma<T>::run(acc[2 * dp + 1], pa, v2 & mk0, v3 & mk1);
                }
            }
            __syncwarp();
            if (lane == 0)
                dev::mbar_arrive(dev::smem_addr(&c.empty[st]));
        }
        if (!alive)
            break;

        // ---- merge the four consumer warps ----
        lrow0 += __shfl_xor_sync(0xffffffffu, lrow0, 1);
        lrow0 += __shfl_xor_sync(0xffffffffu, lrow0, 2);
        lrow1 += __shfl_xor_sync(0xffffffffu, lrow1, 1);
        lrow1 += __shfl_xor_sync(0xffffffffu, lrow1, 2);
        float *mine = c.macc + warp * rows_cap * SA;
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
            c.mml[(warp * kHeadsPerItem + r0) * 2] = (live0 && lrow0 > 0.f) ? mrow0 : -INFINITY;
            c.mml[(warp * kHeadsPerItem + r0) * 2 + 1] = lrow0;
            c.mml[(warp * kHeadsPerItem + r0 + 8) * 2] = (live1 && lrow1 > 0.f) ? mrow1 : -INFINITY;
            c.mml[(warp * kHeadsPerItem + r0 + 8) * 2 + 1] = lrow1;
        }
        }
#ifdef PA_TRACE
        const unsigned long long t_m0 = trace_clock();
#endif
        if (merge_pfx) {
            if (!pfx_ready) {  // first prefix row of this CTA: wait for pass 1 once
                dev::grid_dependency_wait();
                pfx_ready = true;
                stage_prefix<D>(p, it, pfx_s, threadIdx.x);
            }
            dev::cp_async_wait_all();
        }
        if (threadIdx.x == 0)
            probe_split_last(p, it, c);
        if (!consumer_sync(p, c, sph)) {
            break;
        }
        finalize_item<T, D, kShare>(p, it, c.macc, c.mml, rows_cap, threadIdx.x, pfx_s, *c.merge == 2);
        if (!finish_item<T, D, kShare>(p, it, c, sph, warp, lane, pfx_s)) {
            break;
        }
#ifdef PA_TRACE
        if (threadIdx.x == 0) {
            PA_TRACE_ADD(9, trace_clock() - t_m0);
            if (p.balanced && it.partial && *c.merge)
                PA_TRACE_ADD(10, 1);
        }
#endif
        if (*c.abort)
            break;
    }
    // after an early stop, prefix-row copies this thread started land before it exits
    if constexpr (kShare)
        dev::cp_async_wait_all();
#ifdef PA_TRACE
    if (threadIdx.x == 0)
        PA_TRACE_SET(2, dev::global_timer_ns());
#endif
}

// ---------------------------------------------------------------------------
// fp32 partition kernel: CUDA-core consumers (same producer, ring and merge).
// H: query rows an item of the launch carries at most (1, 4 or 16).  The
// consumers' per-row state and loops are sized by it: a launch whose items hold
// one row (multi-head attention) carries no predicated-off work for fifteen
// others and keeps its state in registers.
// ---------------------------------------------------------------------------
template <int D, int BS, int H, int kMode>
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
    static_assert(H == 1 || H == 4 || H == kHeadsPerItem, "row capacities 1, 4, 16");
    constexpr int SA = D + kAccPad;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int rows_cap = item_rows_cap(p);
    constexpr bool kShare = kMode == kModePrefix || kMode == kModeOwn;
    const int pfx_rows = kShare ? item_pfx_rows(p) : 0;
    const SmemLayout lay =
        make_layout(C::kStages, C::kStageBytes, rows_cap, D, sizeof(float), pfx_rows);
    const CtaState c = cta_state(smem, lay, C::kStages);
    init_cta(p, c, C::kStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (warp == kConsumerWarps) {
        producer_loop<float, D, BS, C::kBPS, C::kChunks, C::kTileBytes, C::kStages, kMode,
                      kCopyRuntime>(p, &tmap_k, &tmap_v, c, lane);
        return;
    }

    const int t = lane % BS;
    const int part = lane / BS;
    uint32_t g = 0;
    uint32_t sph = 0;
#ifdef PA_TRACE
    if (threadIdx.x == 0) {
        unsigned int smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        PA_TRACE_SET(0, dev::global_timer_ns());
        PA_TRACE_SET(8, smid);
    }
#endif
    bool pfx_ready = !kShare || !defers_dependency(p);  // prefix rows may be read
    for (uint32_t n = 0;; ++n) {
        const uint32_t slot = n % kItemSlots;
        if (!warp_wait(p, c, &c.item_full[slot], (n / kItemSlots) & 1u)) {
            break;
        }
        const Item it = load_item(&c.items[slot]);
        if (it.seq < 0)
            break;
        // a planned first item takes its length from the plan: its append is stored
        // only if that is the length the launch reads (read here, used stages later)
        const bool append_ok = (kMode != kModePlan && (kMode != kModeOwn || p.plan == nullptr)) ||
                               p.k_new == nullptr || clamp_len(p, it.tseq, BS) == it.len;
        const bool merge_pfx = kShare && (it.flags() & kMergePrefix) != 0;
        float *pfx_s = c.pfx + (n & 1) * pfx_rows * (D + kPfxPad);
        if (merge_pfx && pfx_ready)
            stage_prefix<D>(p, it, pfx_s, threadIdx.x);
        const float *qs = reinterpret_cast<const float *>(c.qslots) + slot * kHeadsPerItem * D;

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
        bool alive = true;
        const int rot = it.rot();
        for (int j = it.j0; j < it.j1; ++j, ++g) {
            if ((j - it.j0 + rot) % kConsumerWarps != warp)
                continue;
            const uint32_t st = g % C::kStages;
#ifdef PA_TRACE
            const unsigned long long t_sw = trace_clock();
#endif
            if (!warp_wait(p, c, &c.full[st], (g / C::kStages) & 1u)) {
                alive = false;
                break;
            }
#ifdef PA_TRACE
            if (threadIdx.x == 0) {
                const unsigned long long t_now = trace_clock();
                PA_TRACE_ADD(13, t_now - t_sw);
                PA_TRACE_SET(11, t_now);
                if (trace_first_tile(p.pass))
                    PA_TRACE_SET(1, t_now);
            }
#endif
            const int valid = min(BS, it.len - j * BS);
            static_assert(C::kBPS == 1, "fp32 stages hold one block");
            const uint8_t *kt = c.ring + (size_t)st * C::kStageBytes;
            const uint8_t *vt = kt + C::kBlockTile;
            if (c.newinfo[2 * st] >= 0)
                patch_newest_row<float, D, BS>(p, it, c, st, c.ring + (size_t)st * C::kStageBytes,
                                               lane, append_ok);

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
                dev::mbar_arrive(dev::smem_addr(&c.empty[st]));
        }
        // the query rows of this slot are no longer read (every read of them fed an
        // FMA above); the descriptor fields are settled like the fp16/bf16 path's
        {
            const uint32_t all = __reduce_xor_sync(
                0xffffffffu, (uint32_t)(it.seq ^ it.kvh ^ it.hg ^ it.len ^ it.j0 ^ it.j1 ^
                                        it.qrow0 ^ it.rows ^ it.partial ^ it.prow0 ^ it.tseq ^
                                        it.packed ^ it.c_first ^ it.nparts) ^
                                  it.total_lo ^ it.total_hi);
            if (lane == 0)
                dev::settle_loads(&c.sink[warp], all);
        }
        __syncwarp();
        if (lane == 0)
            dev::mbar_arrive(dev::smem_addr(&c.item_empty[slot]));
        if (!alive)
            break;

        float *mine = c.macc + warp * rows_cap * SA;
#pragma unroll
        for (int r = 0; r < H; ++r) {
            if (r < it.rows) {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    mine[r * SA + lane * VEC + e] = acc[r][e];
                if (lane == 0) {
                    c.mml[(warp * kHeadsPerItem + r) * 2] = lr[r] > 0.f ? mr[r] : -INFINITY;
                    c.mml[(warp * kHeadsPerItem + r) * 2 + 1] = lr[r];
                }
            }
        }
        if (merge_pfx) {
            if (!pfx_ready) {  // first prefix row of this CTA: wait for pass 1 once
                dev::grid_dependency_wait();
                pfx_ready = true;
                stage_prefix<D>(p, it, pfx_s, threadIdx.x);
            }
            dev::cp_async_wait_all();
        }
#ifdef PA_TRACE
        const unsigned long long t_m0 = trace_clock();
        if (threadIdx.x == 0)
            PA_TRACE_SET(12, t_m0);  // warp 0 done with the item's stages
#endif
        if (threadIdx.x == 0)
            probe_split_last(p, it, c);
        if (!consumer_sync(p, c, sph)) {
            break;
        }
#ifdef PA_TRACE
        if (threadIdx.x == 0)
            PA_TRACE_SET(10, trace_clock());  // all warps done
#endif
        finalize_item<float, D, kShare>(p, it, c.macc, c.mml, rows_cap, threadIdx.x, pfx_s,
                                *c.merge == 2);
        if (!finish_item<float, D, kShare>(p, it, c, sph, warp, lane, pfx_s)) {
            break;
        }
#ifdef PA_TRACE
        if (threadIdx.x == 0)
            PA_TRACE_ADD(9, trace_clock() - t_m0);
#endif
        if (*c.abort)
            break;
    }
    // after an early stop, prefix-row copies this thread started land before it exits
    if constexpr (kShare)
        dev::cp_async_wait_all();
#ifdef PA_TRACE
    if (threadIdx.x == 0)
        PA_TRACE_SET(2, dev::global_timer_ns());
#endif
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
    // launched as a programmatic dependent of the partition kernel: its partials
    // are complete and visible only after this wait
    dev::grid_dependency_wait();
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
// The kernel instance a launch takes: plain decode (walked or planned), or one of
// the shared-prefix decode's two launches (walked or planned alike).
inline int launch_mode(const DecodeParams &p)
{
    if (p.share != nullptr)
        return p.pass == 1 ? kModePrefix : kModeOwn;
    return p.plan != nullptr ? kModePlan : kModePlain;
}

// Items of at most 8 query rows (group <= 8) take the transposed-product
// consumers; wider items the 16-row form.  Caches placed for the joint tensor map
// take the instance that copies K and V together.
template <typename T, int D, int BS>
struct KernelOf {
    template <int kMode, int kCopy>
    static void *pick_copy(const DecodeParams &p)
    {
        return p.group <= kNarrowRows
                   ? reinterpret_cast<void *>(&pa_decode_mma_kernel<T, D, BS, true, kMode, kCopy>)
                   : reinterpret_cast<void *>(&pa_decode_mma_kernel<T, D, BS, false, kMode, kCopy>);
    }
    template <int kMode>
    static void *pick(const DecodeParams &p)
    {
        return p.kv_joint ? pick_copy<kMode, kCopyJoint>(p) : pick_copy<kMode, kCopySplit>(p);
    }
    static void *get(const DecodeParams &p)
    {
        const int mode = launch_mode(p);
        return mode == kModeOwn ? pick<kModeOwn>(p)
               : mode == kModePrefix ? pick<kModePrefix>(p)
               : mode == kModePlan ? pick<kModePlan>(p)
                                     : pick<kModePlain>(p);
    }
};
template <int D, int BS>
struct KernelOf<float, D, BS> {
    // by the launch's row capacity (its widest item)
    template <int kMode>
    static void *pick(const DecodeParams &p)
    {
        const int rows_cap = item_rows_cap(p);
        return rows_cap <= 1
                   ? reinterpret_cast<void *>(&pa_decode_f32_kernel<D, BS, 1, kMode>)
               : rows_cap <= 4
                   ? reinterpret_cast<void *>(&pa_decode_f32_kernel<D, BS, 4, kMode>)
                   : reinterpret_cast<void *>(&pa_decode_f32_kernel<D, BS, kHeadsPerItem, kMode>);
    }
    static void *get(const DecodeParams &p)
    {
        const int mode = launch_mode(p);
        return mode == kModeOwn ? pick<kModeOwn>(p)
               : mode == kModePrefix ? pick<kModePrefix>(p)
               : mode == kModePlan ? pick<kModePlan>(p)
                                     : pick<kModePlain>(p);
    }
};

template <typename T, int D, int BS>
inline size_t smem_bytes_for(int rows, int pfx_rows = 0)
{
    using C = Cfg<T, D, BS>;
    rows = rows < kHeadsPerItem ? rows : kHeadsPerItem;
    return make_layout(C::kStages, C::kStageBytes, rows, D, sizeof(T), pfx_rows).total;
}

int cached_occupancy(void *kernel, int device, size_t smem, size_t max_smem);

// The persistent grid of a launch: its kernel instance's resident CTAs per SM (at
// most kMaxCtasPerSm) times the SMs, or L.grid if that is smaller; 0 if the
// configuration cannot launch.  pa_decode_plan sizes its plan with the same count.
template <typename T, int D, int BS>
long long persistent_grid(const DecodeLaunch &L, void *kern, size_t smem, cudaError_t *err)
{
    const size_t smem_max = smem_bytes_for<T, D, BS>(kHeadsPerItem, kHeadsPerItem);
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess)
        return 0;
    const int per_sm = cached_occupancy(kern, dev, smem, smem_max);
    if (per_sm <= 0)
        return 0;
    long long grid = (long long)min(per_sm, kMaxCtasPerSm) * L.sm_count;
    if (L.grid > 0 && L.grid < grid)
        grid = L.grid;
    return grid;
}

template <typename T, int D, int BS>
int plan_grid_impl(const DecodeLaunch &L)
{
    void *kern = KernelOf<T, D, BS>::get(L.p);
    const size_t smem = smem_bytes_for<T, D, BS>(item_rows_cap(L.p), item_pfx_rows(L.p));
    cudaError_t e = cudaSuccess;
    return (int)persistent_grid<T, D, BS>(L, kern, smem, &e);
}

template <typename T, int D, int BS>
cudaError_t launch_decode_impl(const DecodeLaunch &L, cudaStream_t stream)
{
    const DecodeParams &p = L.p;
    void *kern = KernelOf<T, D, BS>::get(p);
    const size_t smem = smem_bytes_for<T, D, BS>(item_rows_cap(p), item_pfx_rows(p));
    cudaError_t e = cudaSuccess;
    long long grid = persistent_grid<T, D, BS>(L, kern, smem, &e);
    if (e != cudaSuccess)
        return e;
    if (grid <= 0)
        return cudaErrorInvalidConfiguration;
    if (!p.balanced) {
        const long long items =
            (long long)p.num_seqs * p.max_parts * p.num_kv_heads * p.head_groups;
        if (grid > items)
            grid = items;
    }
    if (grid < 1)
        grid = 1;
    // a planned launch runs on exactly the grid its plan has an entry per CTA of
    if (p.plan != nullptr && grid != L.grid)
        return cudaErrorInvalidConfiguration;
    void *args[] = {const_cast<DecodeParams *>(&L.p), const_cast<CUtensorMap *>(&L.tmap_k),
                    const_cast<CUtensorMap *>(&L.tmap_v)};
    // Both kernels are programmatic dependents of whatever precedes them in the
    // stream: their launch and prologue overlap the previous kernel's tail, and
    // griddepcontrol.wait orders every read of the previous kernel's results.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    #ifdef PA_NO_PDL
    attr[0].val.programmaticStreamSerializationAllowed = 0;
#else
    attr[0].val.programmaticStreamSerializationAllowed = 1;
#endif
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, kern, args);
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t mcfg = {};
    mcfg.blockDim = dim3(128);
    mcfg.dynamicSmemBytes = 0;
    mcfg.stream = stream;
    mcfg.attrs = attr;
    mcfg.numAttrs = 1;
    if (!p.balanced && p.max_parts > 1) {
        mcfg.gridDim = dim3((unsigned)((p.num_q_heads + 3) / 4), (unsigned)p.num_seqs);
        e = cudaLaunchKernelEx(&mcfg, pa_merge_kernel<T, D>, p, (int)BS);
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
int plan_grid_dispatch(const DecodeLaunch &L)
{
    if (L.head_dim == 128 && L.block_size == 16)
        return plan_grid_impl<T, 128, 16>(L);
    if (L.head_dim == 128 && L.block_size == 32)
        return plan_grid_impl<T, 128, 32>(L);
    if (L.head_dim == 64 && L.block_size == 16)
        return plan_grid_impl<T, 64, 16>(L);
    if (L.head_dim == 64 && L.block_size == 32)
        return plan_grid_impl<T, 64, 32>(L);
    return 0;
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

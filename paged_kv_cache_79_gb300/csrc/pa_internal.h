// Internal declarations shared by the translation units of libpagedkv.so.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pagedkv.h"

namespace pagedkv {

// Query heads handled by one work item: the M dimension of the m16n8k16 tiles.
constexpr int kHeadsPerItem = 16;
// Consumer warps per CTA; one more warp issues the TMA copies.
constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
// A device-side wait gives up after this long (ns) and raises an error flag.  The
// limit a launch uses is DecodeParams::wait_ns (pa_set_wait_limit_ns); the wait for
// copies still in flight when a CTA stops early always takes this one.
constexpr unsigned long long kWaitTimeoutNs = PA_WAIT_LIMIT_DEFAULT_NS;

// Everything the decode kernels read besides the two tensor maps.
struct DecodeParams {
    void *out;                    // [S][Hq][D] storage dtype
    const void *q;                // [S][Hq][D] storage dtype
    const int32_t *block_tables;  // [S][max_blocks]
    const int32_t *context_lens;  // [S]
    // Partial results (fp32 output rows and their log2-sum-exp), null when unused:
    //   fixed partitions: rows [S][max_parts][Hq];  balanced split: rows [2*grid][16]
    float *part_o;
    float *part_lse;
    unsigned int *errors;         // device error flags (PA_DEVERR_*)
    float scale_log2;             // softmax scale * log2(e)
    int num_seqs;
    int max_blocks;               // block-table row length
    int num_blocks;               // physical blocks in the pool
    int num_q_heads;
    int num_kv_heads;
    int group;                    // num_q_heads / num_kv_heads
    int head_groups;              // ceil(group / kHeadsPerItem)
    int partition_blocks;         // fixed partitions: blocks per partition
    int max_parts;                // fixed partitions: ceil(max_blocks / partition_blocks)
    int balanced;                 // 1: balanced split over the persistent grid
    unsigned int epoch;           // balanced split: tag of this call's merge counters
    unsigned long long *counters; // balanced split: [grid] (epoch << 32 | partials written)
    // Fused append (null when off): the newest token of every sequence (position
    // context_len - 1) takes its K/V rows from k_new/v_new [S][Hkv][D] instead of the
    // cache, and the kernel writes them into the cache at that position's slot.
    const void *k_new;
    const void *v_new;
    void *k_cache;
    void *v_cache;
    // Shared-prefix decode (null share: off).  share[s] = {first member of s's
    // group, shared leading blocks}; pass 1 streams each group's shared blocks once
    // for all members and writes fp32 rows + log2-sum-exp to pfx
    // ([S][Hq][D], [S][Hq]); pass 0 then covers each sequence's own blocks and merges.
    const int32_t *share;
    int pass;
    float *pfx;  // rows of head_dim + 4 floats: the row's o, then its log2-sum-exp
    // Limit of every bounded wait of the launch (ns), but for the drain of copies in
    // flight; kWaitTimeoutNs unless pa_set_wait_limit_ns changed it.
    unsigned long long wait_ns;
    // Plain balanced-split decode: kPlanInts per CTA of the host-computed start
    // (pa_decode_plan), or null to walk the stream on the device.
    const int32_t *plan;
    // 1: the K tensor map spans both caches (a fifth dimension of extent 2 steps from
    // K to V), so one copy fetches a block's K and V tiles; 0: one copy per cache.
    int kv_joint;
};

// The wait limit decode launches take (pa_set_wait_limit_ns).
unsigned long long wait_limit_ns();

// Balanced split: partial slots are reserved for at most this many CTAs per SM.
constexpr int kMaxCtasPerSm = 4;

// Schedule constants shared by the kernels and the host-side plan
// (pa_decode_plan), which replays the balanced split's walk.
#ifndef PA_STAGE_TOKENS
#define PA_STAGE_TOKENS 32  // tokens per ring stage (fp16/bf16): blocks of 16 go two per stage
#endif
#ifndef PA_UNIT_COST
#define PA_UNIT_COST 4      // stream positions charged per unit for its fixed cost
#endif
#ifndef PA_MIN_POSITIONS
#define PA_MIN_POSITIONS 4  // stream positions per CTA at least
#endif
constexpr int kUnitCost = PA_UNIT_COST;
constexpr long long kMinPositions = PA_MIN_POSITIONS;
static_assert(kUnitCost >= 1, "every unit needs a start position");

// Blocks per ring stage of the partition kernel for a storage type of elem_bytes.
inline int blocks_per_stage(int elem_bytes, int block_size)
{
    return (elem_bytes == 4 || PA_STAGE_TOKENS <= block_size) ? 1 : PA_STAGE_TOKENS / block_size;
}

// Balanced split: positions per CTA at least -- kMinPositions, or, for a batch of
// short units (8 positions or fewer on average), the average unit -- and the CTAs
// a stream of `total` positions is spread over (at most `grid`).
__host__ __device__ __forceinline__ int balanced_divisor(long long total, long long units)
{
    const long long avg = units > 0 ? (total + units - 1) / units : 1;
    return (int)(avg <= 8 && avg > kMinPositions ? avg : kMinPositions);
}
__host__ __device__ __forceinline__ long long balanced_grid_of(long long total, int divisor, long long grid)
{
    const long long g = (total + divisor - 1) / divisor;
    return g < 1 ? 1 : (g < grid ? g : grid);
}

// Host-computed start of each CTA of a balanced-split launch (pa_decode_plan):
// kPlanInts int32 per CTA of the persistent grid, in this order.
constexpr int kPlanInts = 32;
enum PlanField {
    kPlanSeq = 0,       // sequence whose positions hold the CTA's first position
    kPlanBase = 1,      // first position of that sequence (int64: lo, hi)
    kPlanLen = 3,       // its context length, clamped to the table
    kPlanTotal = 4,     // positions of the whole stream (int64: lo, hi)
    kPlanDiv = 6,       // positions per CTA at least
    kPlanG = 7,         // CTAs the stream is spread over
    kPlanGrid = 8,      // persistent grid the plan was made for
    kPlanStart = 9,     // the CTA's range [start, end) (int64 each: lo, hi)
    kPlanEnd = 11,
    kPlanJ0 = 13,       // first block of the CTA's first item
    kPlanSeqs = 14,     // batch size the plan was made for
    kPlanAux = 15,      // shared-prefix passes: see kAux* below
    kPlanBlocks = 16,   // block ids j0 .. j0 + 15 of the first item's sequence (-1 past it)
};
constexpr int kPlanWindow = kPlanInts - kPlanBlocks;
// kPlanAux of a shared-prefix pass's plan: the first sequence's units beyond its
// length -- pass 1: the members of its group; pass 0: the first block of its own
// units -- in the low bits, and two flags.
constexpr int kAuxValueMask = (1 << 29) - 1;
constexpr int kAuxUnitMajor = 1 << 29;  // pass 0 streams in (unit, sequence) order
constexpr int kAuxShareErr = 1 << 30;   // the first sequence ends inside its shared blocks

struct DecodeLaunch {
    DecodeParams p;
    CUtensorMap tmap_k;  // K, or K and V together when p.kv_joint
    CUtensorMap tmap_v;
    int head_dim;
    int block_size;
    int grid;                     // 0: let the launcher size it from occupancy
    int sm_count;
};

// Persistent grid (CTAs) of a balanced-split launch of the plain decode with a
// plan; 0 if the configuration cannot launch.
int plan_grid_f32(const DecodeLaunch &L);
int plan_grid_f16(const DecodeLaunch &L);
int plan_grid_bf16(const DecodeLaunch &L);

// Per-dtype launchers (pa_decode_{f32,f16,bf16}.cu).  They size the persistent
// grid from occupancy, launch the partition kernel and, when any sequence can
// span several partitions, the merge kernel.
cudaError_t launch_decode_f32(const DecodeLaunch &L, cudaStream_t stream);
cudaError_t launch_decode_f16(const DecodeLaunch &L, cudaStream_t stream);
cudaError_t launch_decode_bf16(const DecodeLaunch &L, cudaStream_t stream);

// Shared-memory bytes the partition kernel needs (including alignment slack).
size_t decode_smem_bytes_f32(int head_dim, int block_size, int group);
size_t decode_smem_bytes_f16(int head_dim, int block_size, int group);
size_t decode_smem_bytes_bf16(int head_dim, int block_size, int group);

// Resident CTAs per SM of `kernel` with `smem` dynamic shared memory on `device`
// (raises the kernel's dynamic shared-memory limit to `max_smem` first).  Cached.
int cached_occupancy(void *kernel, int device, size_t smem, size_t max_smem);

// Number of SMs of `device` (cached).
int sm_count(int device);

// Record `e` as this thread's last CUDA error (read by pa_last_cuda_error) and
// clear the runtime's sticky launch error.
void note_cuda_error(cudaError_t e);

cudaError_t launch_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                                     const int64_t *slots, int num_tokens, size_t row_bytes,
                                     long long num_slots, cudaStream_t stream);
cudaError_t launch_move_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                               const int32_t *src_ids, int src_stride, const int32_t *dst_ids,
                               int dst_stride, int num, int src_blocks, int dst_blocks,
                               size_t block_bytes, cudaStream_t stream);
cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int32_t *pairs, int num_pairs,
                               int num_blocks, size_t block_bytes, cudaStream_t stream);

}  // namespace pagedkv

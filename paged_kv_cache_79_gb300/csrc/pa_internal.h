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
};

// The wait limit decode launches take (pa_set_wait_limit_ns).
unsigned long long wait_limit_ns();

// Balanced split: partial slots are reserved for at most this many CTAs per SM.
constexpr int kMaxCtasPerSm = 4;

struct DecodeLaunch {
    DecodeParams p;
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    int head_dim;
    int block_size;
    int grid;                     // 0: let the launcher size it from occupancy
    int sm_count;
};

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

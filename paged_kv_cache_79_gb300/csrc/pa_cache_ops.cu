// Cache writes: KV append through a slot mapping, and whole-block moves: the
// copy-on-write copy within one pool, swapping between the device pool and a pool
// in pinned host memory, and packing blocks into (or out of) a contiguous staging
// buffer for a KV transfer.
//
// reshape_and_cache follows CSDN tutorial "PagedAttention实战" §3.1 append_kv
// (token position -> logical page pos // page_size, offset pos % page_size; the
// allocator turns that into a slot = physical_block * B + offset).  copy_blocks is
// the copy half of copy-on-write ("Efficient Memory Management for LLM Serving with
// PagedAttention", azimuth.plus summary, section "Memory sharing"); swapping is the
// same summary's section "vLLM" (preempted requests' blocks move to CPU memory);
// staging follows the bidirectional KV-transfer article (spke.com translation of
// an AWS blog post on prefill/decode-disaggregated vLLM), section "Bidirectional KV
// transfer".  All are plain 16-byte vector copies: the cost is launch latency and
// the bytes moved.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pagedkv {

namespace {

// One CTA per (token, K or V).  A token's row of num_kv_heads * head_dim elements is
// contiguous both in the input and in the cache ([NB][B][Hkv][d] layout).
__global__ void __launch_bounds__(128)
    reshape_and_cache_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                             uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                             const int64_t *__restrict__ slots, int vec_per_row, long long num_slots)
{
    dev::grid_dependency_wait();  // the cache and the inputs may come from the previous kernel
    dev::grid_launch_dependents();
    const int t = blockIdx.x;
    const int64_t slot = slots[t];
    if (slot < 0 || slot >= num_slots)
        return;
    const uint4 *src = (blockIdx.y == 0 ? k : v) + (size_t)t * vec_per_row;
    uint4 *dst = (blockIdx.y == 0 ? k_cache : v_cache) + (size_t)slot * vec_per_row;
    for (int i = threadIdx.x; i < vec_per_row; i += blockDim.x)
        dst[i] = __ldg(src + i);
}

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

// Block i of the call moves from block src_ids[i * src_stride] of the source pool
// to block dst_ids[i * dst_stride] of the destination pool; a null id array means
// block i itself (a contiguous staging buffer).  Either pool may be pinned host
// memory (reached through unified addressing).  Out-of-range ids skip the block.
// grid = (blocks, 2 caches, chunks of kCopyThreads * kCopyUnroll 16-byte vectors)
__global__ void __launch_bounds__(kCopyThreads)
    move_blocks_kernel(const uint4 *src_k, const uint4 *src_v, uint4 *dst_k, uint4 *dst_v,
                       const int32_t *__restrict__ src_ids, int src_stride,
                       const int32_t *__restrict__ dst_ids, int dst_stride, int src_blocks,
                       int dst_blocks, long long vec_per_block)
{
    dev::grid_dependency_wait();
    dev::grid_launch_dependents();
    const int i = blockIdx.x;
    const int src = src_ids ? src_ids[(size_t)i * src_stride] : i;
    const int dst = dst_ids ? dst_ids[(size_t)i * dst_stride] : i;
    if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks)
        return;
    const uint4 *s = (blockIdx.y == 0 ? src_k : src_v) + (size_t)src * vec_per_block;
    uint4 *d = (blockIdx.y == 0 ? dst_k : dst_v) + (size_t)dst * vec_per_block;
    const long long first = (long long)blockIdx.z * kCopyThreads * kCopyUnroll + threadIdx.x;
    uint4 tmp[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const long long j = first + (long long)u * kCopyThreads;
        if (j < vec_per_block)
            tmp[u] = s[j];
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const long long j = first + (long long)u * kCopyThreads;
        if (j < vec_per_block)
            d[j] = tmp[u];
    }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                                     const int64_t *slots, int num_tokens, size_t row_bytes,
                                     long long num_slots, cudaStream_t stream)
{
    const int vec = (int)(row_bytes / 16);
    const int threads = vec >= 128 ? 128 : (vec >= 64 ? 64 : 32);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    #ifdef PA_NO_PDL
    attr[0].val.programmaticStreamSerializationAllowed = 0;
#else
    attr[0].val.programmaticStreamSerializationAllowed = 1;
#endif
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_tokens, 2);
    cfg.blockDim = dim3(threads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, reshape_and_cache_kernel, static_cast<const uint4 *>(k),
                              static_cast<const uint4 *>(v), static_cast<uint4 *>(k_cache),
                              static_cast<uint4 *>(v_cache), slots, vec, num_slots);
}

cudaError_t launch_move_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                               const int32_t *src_ids, int src_stride, const int32_t *dst_ids,
                               int dst_stride, int num, int src_blocks, int dst_blocks,
                               size_t block_bytes, cudaStream_t stream)
{
    const long long vec = (long long)(block_bytes / 16);
    const long long per_cta = (long long)kCopyThreads * kCopyUnroll;
    const unsigned z = (unsigned)((vec + per_cta - 1) / per_cta);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
#ifdef PA_NO_PDL
    attr[0].val.programmaticStreamSerializationAllowed = 0;
#else
    attr[0].val.programmaticStreamSerializationAllowed = 1;
#endif
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num, 2, z);
    cfg.blockDim = dim3(kCopyThreads);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, move_blocks_kernel, static_cast<const uint4 *>(src_k),
                              static_cast<const uint4 *>(src_v), static_cast<uint4 *>(dst_k),
                              static_cast<uint4 *>(dst_v), src_ids, src_stride, dst_ids, dst_stride,
                              src_blocks, dst_blocks, vec);
}

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int32_t *pairs, int num_pairs,
                               int num_blocks, size_t block_bytes, cudaStream_t stream)
{
    return launch_move_blocks(k_cache, v_cache, k_cache, v_cache, pairs, 2, pairs + 1, 2, num_pairs,
                              num_blocks, num_blocks, block_bytes, stream);
}

}  // namespace pagedkv

// pa_decode_noalloc: pa_decode whose split-KV scratch lives in a fixed device array.
//
// Some callers cannot hand pa_decode a workspace: code that runs under an engine or
// framework which has already planned every device buffer and forbids allocation
// once it is running (an inference-engine plugin's enqueue, an embedded runtime with
// a static memory budget), or a plain C caller that has no device allocator of its
// own and must not call cudaMalloc on its hot path (cudaMalloc can synchronise the
// device and stalls other streams).  For them this entry point takes no workspace:
// the partial results of long sequences go to g_noalloc_scratch, a file-scope
// __device__ array of PA_DECODE_NOALLOC_SCRATCH_BYTES.  Nothing here calls
// cudaMalloc, cudaFree or any allocating library routine.
//
// Host code never uses the array's name as an address (on the host it is only a
// stand-in): the first call on each device, with that device current, looks its
// device address up with cudaGetSymbolAddress and caches it.
#include <mutex>

#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch on each device

// Set-up, once per device, with `device` current.
cudaError_t scratch_address(int device, void **out)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[device]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return cudaSuccess;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void *out, const void *q, const void *k_cache,
                                       const void *v_cache, const int32_t *block_tables,
                                       int max_blocks_per_seq, const int32_t *context_lens,
                                       int num_seqs, int num_blocks, float scale, int num_q_heads,
                                       int num_kv_heads, int head_dim, int block_size,
                                       pa_dtype dtype, int partition_size, void *stream)
{
    const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 block_size, max_blocks_per_seq, partition_size);
    if (need == (size_t)-1 || num_seqs == 0)  // let pa_decode report the argument error
        return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                         num_seqs, num_blocks, scale, num_q_heads, num_kv_heads, head_dim,
                         block_size, dtype, partition_size, nullptr, 0, stream);
    if (need > (size_t)PA_DECODE_NOALLOC_SCRATCH_BYTES)
        return PA_ERR_UNSUPPORTED;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && (dev < 0 || dev >= kMaxDevices))
        return PA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (e == cudaSuccess)
        e = scratch_address(dev, &scratch);
    if (e != cudaSuccess) {
        pagedkv::note_cuda_error(e);
        return PA_ERR_CUDA;
    }
    return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, num_blocks, scale, num_q_heads, num_kv_heads, head_dim, block_size,
                     dtype, partition_size, scratch, (size_t)PA_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
